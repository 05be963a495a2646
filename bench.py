#!/usr/bin/env python
"""Benchmark of the QSA token-indexer hot path (pool -> score -> select) on GB300.

Workload (one bench step = one decode step of one sequence): batch-1 decode at
64k context -- one query row at positions 65280..65535 (16384 blocks), the
pooled block keys cached, the block a token completes pooled on that step, then
score and select with budget 2048.  To keep every step's inputs out of L2, the
steps rotate over R independent sequences whose key caches together exceed the
129 MB L2 (no flush is needed).  Step k decodes position 65280 + (k mod 256) of
sequence k mod R with R odd, so consecutive steps walk consecutive positions
and every fourth step completes a block and pools it.  Steps are replayed from
CUDA graphs, so the host does not pace the GPU.

Printed: one JSON line (rank 0) with rows/s, per-kernel roofline of the
dominant kernel (CUDA events, live), the oracle's CPU baseline, an end-to-end
number through the public entry point with host buffers, clocks sampled during
the timed region, and secondary measurements (selection at 256k).

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import qsa_inputs as qi  # noqa: E402

METRIC = "indexer rows/s (pool+score+select) at 64k ctx; select µs/row at 256k; % roofline"
WORKLOAD = "decode batch 1, pos 65280..65535 of a 64k-token context (16384 blocks), budget 2048"
TOKENS = 65536
N_BLOCKS = TOKENS // 4
FIRST_POS = TOKENS - 256
BUDGET = 2048
EPS = 1e-6
THETA = 10000.0
L2_BYTES = 129 * 1024 * 1024

# algorithmic bytes per unit: what each kernel must move at minimum (HBM-bound kernels)
POOL_BYTES_PER_BLOCK = 1024 + 256 + 256
SCORE_BYTES_PER_BLOCK = 256 + 4
SELECT_BYTES_PER_BLOCK = 4          # + 1 byte per mask token written
GATHER_WIDTH = 512                  # 2 KV heads x head dim 256, bf16
GATHER_PAGE = 16                    # tokens per cache page
GATHER_BYTES_PER_TOKEN = 8 * GATHER_WIDTH + 8   # K, V read and written; index and page entry
DECODE_FUSED_SOURCES = ("qsa_decode.cu", "qsa_tc_device.cuh", "qsa_select_util.cuh", "qsa_device.cuh", "qsa_tma.h",
                        "qsa_launch.h")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=16384)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=1024)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ncu-case", default=None,
                    help="run one small case of a kernel for an ncu capture and exit")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def source_digest(names) -> str:
    """sha256 (12 hex) over a kernel's source files, concatenated in order."""
    h = hashlib.sha256()
    for name in ([names] if isinstance(names, str) else names):
        with open(os.path.join(ROOT, "sparse_attention_token_qsa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def recorded_traffic(kernel: str, workload: str, src: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is
    unchanged since that capture (profiles/dram_traffic.txt)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(src)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[3] == digest:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples while the timed region runs (host wall clock stamps)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            time.sleep(0.2)
            if self.proc.poll() not in (None, 0) and gpu_id:   # id not accepted: all GPUs
                self.proc = subprocess.Popen(cmd[:-2] + ["-i", "0"], stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def summary(self, t0: float, t1: float):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        inside = [s for t, s in self.samples if t0 <= t <= t1 + 0.15]
        if not inside:  # region shorter than the sampling period: nearest samples
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[1]]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        smax = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 4 + i and s[4 + i].lower().startswith("active")})
        power = [num(s[2]) for s in inside if num(s[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "power_w_max": max(power) if power else None, "samples": len(inside)}


def gpu_uuid(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def dev_tensor(torch, a, device):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


# ------------------------------------------------------------ the workload

class DecodeWorkload:
    """R independent 64k-token sequences, each with a raw-key cache, a pooled
    block-key cache, 256 decode query rows, and its own score and mask rows."""

    def __init__(self, torch, qsa, device, n_seq: int):
        self.torch, self.qsa, self.device = torch, qsa, device
        self.R = n_seq
        rng = qi.rng_for(1)
        self.q_norm_w, self.k_norm_w = qi.norm_weights(rng)
        c, s = qsa.qsa_rope_tables(TOKENS, THETA)
        self.cos_h, self.sin_h = c, s
        self.cos, self.sin = dev_tensor(torch, c, device), dev_tensor(torch, s, device)
        self.qw = dev_tensor(torch, self.q_norm_w, device)
        self.kw = dev_tensor(torch, self.k_norm_w, device)
        self.keys, self.cache, self.q, self.scores, self.mask = [], [], [], [], []
        self.keys_host0 = None
        self.q_host0 = None
        for r in range(n_seq):
            rr = qi.rng_for(1, salt=r + 1)
            k = qi.raw_keys(rr, TOKENS, token_scale=True)
            q = np.ascontiguousarray(qi.fused_qk(rr, 256)[:, :512])
            if r == 0:
                self.keys_host0, self.q_host0 = k, q
            self.keys.append(dev_tensor(torch, k, device))
            self.q.append(dev_tensor(torch, q, device))
            self.cache.append(torch.zeros((N_BLOCKS, 128), dtype=torch.int16, device=device))
            self.scores.append(torch.zeros((1, N_BLOCKS), dtype=torch.float32, device=device))
            self.mask.append(torch.zeros((1, TOKENS), dtype=torch.uint8, device=device))
        self.status = qsa.new_status(device)
        # zeroed workspace of the fused decode entry (every call leaves it zero)
        self.dws = qsa.new_decode_workspace(1, TOKENS, device)
        # every block of the sequence is cached before the first step; a step
        # that completes a block pools it again (the same key, the same work)
        for r in range(n_seq):
            qsa.qsa_pool_blocks(self.keys[r], 128, 0, N_BLOCKS, self.kw, self.cos, self.sin,
                                TOKENS, EPS, self.cache[r])
        self.positions = dev_tensor(torch, np.arange(FIRST_POS, TOKENS, dtype=np.int32), device)
        torch.cuda.synchronize(device)

    def step_params(self, k: int):
        """Step k: sequence k mod R at position FIRST_POS + (k mod 256).  R is
        odd (coprime to 256), so every run of 4 steps holds one step whose
        token completes a block, and all R * 256 (sequence, position) pairs
        come round before any repeats."""
        seq = k % self.R
        j = k % 256
        return seq, j, FIRST_POS + j

    def pool(self, k):
        seq, j, p = self.step_params(k)
        if (p + 1) % 4 == 0:
            b = (p + 1) // 4 - 1
            self.qsa.qsa_pool_blocks(self.keys[seq][4 * b:], 128, b, 1, self.kw, self.cos,
                                     self.sin, TOKENS, EPS, self.cache[seq])

    def score(self, k):
        seq, j, p = self.step_params(k)
        self.qsa.qsa_score_rows(self.q[seq][j:j + 1], 512, self.positions[j:j + 1], None, 1,
                                TOKENS, self.qw, self.cos, self.sin, TOKENS, EPS, self.cache[seq],
                                None, self.scores[seq], N_BLOCKS, self.status)

    def select(self, k):
        seq, j, p = self.step_params(k)
        self.qsa.qsa_select_mask(self.scores[seq], N_BLOCKS, self.positions[j:j + 1], 1, TOKENS,
                                 BUDGET, self.mask[seq], self.status)

    def step_three(self, k):
        """One step through the three single-stage entry points."""
        self.pool(k)
        self.score(k)
        self.select(k)

    def step(self, k, q_src=None, pos_src=None, pool=True, keys_src=None, mask_dst=None):
        """One decode step through its public entry point (qsa_decode_index_select):
        pool the block the token completes, then score and select in one launch.
        The query row, position, raw keys and mask row may be given in other
        (e.g. pinned host) buffers."""
        seq, j, p = self.step_params(k)
        completes = pool and (p + 1) % 4 == 0
        b = (p + 1) // 4 - 1
        keys = self.keys[seq] if keys_src is None else keys_src
        self.qsa.qsa_decode_index_select(
            keys[4 * b:] if completes else keys, 128, b if completes else 0,
            1 if completes else 0, self.kw, self.q[seq][j:j + 1] if q_src is None else q_src, 512,
            self.positions[j:j + 1] if pos_src is None else pos_src, 1, TOKENS, self.qw, self.cos,
            self.sin, TOKENS, EPS, BUDGET, self.cache[seq], self.scores[seq], N_BLOCKS,
            self.mask[seq] if mask_dst is None else mask_dst, self.status, self.dws)

    def fused_only(self, k):
        self.step(k, pool=False)


def capture_graphs(torch, fn, steps, chunk=256):
    """CUDA graphs replaying fn(k) for k in steps, chunk steps per graph."""
    graphs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    for i in range(0, len(steps), chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for k in steps[i:i + chunk]:
                fn(k)
        graphs.append(g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return graphs


# Cycles the GPU spins before a timed region starts (~100 us at 2 GHz): the host
# queues the region's graphs meanwhile, so the start event times the device's work
# and not the host's submission of the first graph.
LEAD_SPIN_CYCLES = 200_000


def time_graphs(torch, graphs):
    """Device time of one replay of graphs, in ms.  The first graphs are replayed
    once untimed (a graph's first launch also uploads it); every timed step
    rewrites the same outputs from the same inputs, so the replay changes no
    result."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    for g in graphs[:16]:
        g.replay()
    torch.cuda.synchronize()
    torch.cuda._sleep(LEAD_SPIN_CYCLES)
    start.record()
    for g in graphs:
        g.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


# ------------------------------------------------------------ oracle (CPU)

def oracle_decode_rate(seconds: float, max_rows: int | None = None, min_seconds: float = 0.0):
    """The oracle on the host cores: decode steps at 64k on one sequence,
    row-parallel over threads (each thread runs whole steps).  Runs until
    `seconds` have passed, or sooner once `max_rows` rows are done and at least
    `min_seconds` have passed."""
    import oracle

    orc = oracle.Oracle()
    rng = qi.rng_for(1)
    qw, kw = qi.norm_weights(rng)
    rr = qi.rng_for(1, salt=1)
    keys = qi.raw_keys(rr, TOKENS, token_scale=True)
    q = np.ascontiguousarray(qi.fused_qk(rr, 256)[:, :512])
    c, s = orc.rope_table(TOKENS, THETA)
    cache = orc.pool_blocks(keys, 128, 0, N_BLOCKS, kw, c, s, EPS)
    cores = max(1, min(os.cpu_count() or 1, 64))
    caches = [cache.copy() for _ in range(cores)]
    t_start = time.time()
    stop, min_stop = t_start + seconds, t_start + min_seconds
    counts = [0] * cores

    def worker(t):
        sc = np.zeros((1, N_BLOCKS), np.float32)
        j = t
        while True:
            now = time.time()
            if now >= stop or (max_rows is not None and j >= max_rows and now >= min_stop):
                break
            p = FIRST_POS + (j % 256)
            if (p + 1) % 4 == 0:      # pool the block this token completes (own copy)
                b = (p + 1) // 4 - 1
                orc.pool_blocks(keys[4 * b:], 128, b, 1, kw, c, s, EPS, block_keys=caches[t])
            orc.score_rows(q[j % 256:j % 256 + 1], 512, np.array([p], np.int32), 1, TOKENS, qw, c,
                           s, EPS, caches[t], sc, N_BLOCKS)
            orc.select_row(sc[0, :(p + 1) // 4], p, TOKENS, BUDGET)
            counts[t] += 1
            j += cores

    t0 = time.time()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(worker, range(cores)))
    dt = time.time() - t0
    rows = sum(counts)
    return rows / dt, cores, rows, dt


# ------------------------------------------------------------ main arms

def job_rate(torch, ms_local: float, units_local: float, world: int, device):
    """The whole job's time and rate over `world` ranks (weak scaling): the
    slowest rank's time, and the units every rank processed divided by it.
    Ranks hold independent replicas, so these two reductions are the only
    exchange; with one rank they are the local values."""
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    u = torch.tensor([units_local], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    ms = float(t.item())
    return ms, float(u.item()) / (ms / 1000.0)


def run_reference(args, rank, world):
    if rank != 0:
        return
    # at least K decode rows and at least 20 s of work, row-parallel over the
    # host cores, bounded at 240 s of wall time (the line reports how many rows ran)
    rate, cores, rows, dt = oracle_decode_rate(seconds=240.0, max_rows=max(args.steps, 1),
                                               min_seconds=20.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "rows_run": rows, "warmup": args.warmup,
        "ms_per_step": 1000.0 * dt / max(rows, 1) * cores, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": TOKENS, "budget": BUDGET, "rows_per_step": 1,
                   "step_schedule": "row j: position 65280 + j mod 256; a row whose token "
                                    "completes a block pools it",
                   "pool_steps_timed": sum(1 for j in range(rows) if (FIRST_POS + j % 256 + 1) % 4 == 0),
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} decode rows in {dt:.1f} s on {cores} threads"},
        "e2e": {"value": rate, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, device):
    import torch

    import sparse_attention_token_qsa_gb300 as qsa

    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = load_peaks()
    per_seq_bytes = N_BLOCKS * 256 + TOKENS * 256 + N_BLOCKS * 4 + TOKENS
    R = max(9, int(np.ceil(1.5 * L2_BYTES / (N_BLOCKS * 256)))) | 1   # odd: coprime to 256
    wl = DecodeWorkload(torch, qsa, device, R)

    # warm-up (eager): first calls also set kernel attributes outside any capture
    for k in range(max(args.warmup, 3)):
        wl.step(k)
        wl.step_three(k)
    torch.cuda.synchronize()
    code, row = qsa.qsa_read_status(wl.status)
    assert code == 0, f"device status {code} row {row}"

    K = args.steps
    steps = list(range(args.warmup, args.warmup + K))
    graphs = capture_graphs(torch, wl.step, steps)
    for g in graphs[:2]:
        g.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(gpu_uuid(torch, device))
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ms = time_graphs(torch, graphs)
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.summary(t0, t1)
    ms, value = job_rate(torch, ms, K, world, device)  # K rows on every rank
    ms_per_step = ms / K
    pool_steps_timed = sum(1 for k in steps if (wl.step_params(k)[2] + 1) % 4 == 0)
    code, row = qsa.qsa_read_status(wl.status)
    assert code == 0, f"device status {code} row {row}"

    # the same steps through the three single-stage entry points
    g3 = capture_graphs(torch, wl.step_three, steps[:min(K, 4096)])
    three_us = time_graphs(torch, g3) / min(K, 4096) * 1000.0

    # per-kernel durations: the same launches, one kernel at a time, CUDA events
    kern = {}
    for name, fn, bytes_per_launch, src in (
            ("decode_fused", wl.fused_only, SCORE_BYTES_PER_BLOCK * N_BLOCKS + TOKENS,
             DECODE_FUSED_SOURCES),
            ("score", wl.score, SCORE_BYTES_PER_BLOCK * N_BLOCKS, "qsa_score_stream.cu"),
            ("select", wl.select, SELECT_BYTES_PER_BLOCK * N_BLOCKS + TOKENS, "qsa_select.cu")):
        gk = capture_graphs(torch, fn, steps[:min(K, 4096)])
        t_ms = time_graphs(torch, gk) / min(K, 4096)
        kern[name] = {"us": t_ms * 1000.0, "bytes": bytes_per_launch, "src": src}
    pool_steps = [k for k in steps[:4096] if (wl.step_params(k)[2] + 1) % 4 == 0]
    gk = capture_graphs(torch, wl.pool, pool_steps)
    kern["pool"] = {"us": time_graphs(torch, gk) / max(1, len(pool_steps)) * 1000.0,
                    "bytes": POOL_BYTES_PER_BLOCK, "src": "qsa_pool.cu"}
    dom = "decode_fused"
    d = kern[dom]
    achieved = d["bytes"] / (d["us"] * 1e-6) / 1e9
    traffic = recorded_traffic(f"{dom}", "decode64k", d["src"])
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_gbs,
                "unit": "GB/s", "frac": achieved / hbm_gbs, "traffic": traffic,
                "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes": d["bytes"],
                "avg_launch_us": d["us"],
                "note": "batch-1 decode is latency-bound: one 64k row moves "
                        f"{d['bytes'] / 1e6:.2f} MB, {d['bytes'] / (hbm_gbs * 1e3):.2f} us at "
                        "the measured peak, against a launch, a grid barrier and a few "
                        "dependent L2 round trips; the bandwidth-bound kernels' fractions "
                        "are in secondary (score, select, pool, gather)"}
    kernels = {n: {"avg_launch_us": round(v["us"], 3), "algorithmic_bytes": v["bytes"],
                   "achieved_gbs": round(v["bytes"] / (v["us"] * 1e-6) / 1e9, 1),
                   "frac_of_measured_hbm": round(v["bytes"] / (v["us"] * 1e-6) / 1e9 / hbm_gbs, 4)}
               for n, v in kern.items()}

    # end to end through the public decode entry with host buffers: every step's
    # inputs (the query row and position, packed in one 1056-byte record, and
    # the new token's raw key) start in pinned host memory and its mask row ends
    # there.  Two ways of moving them, both timed:
    #  - in place: the kernels read the record and the raw keys, and write the
    #    mask row, directly in pinned host memory over the CPU-GPU link (the
    #    pointers are device-addressable); no copy node;
    #  - copies: one H2D copy of the record and one of the raw key into device
    #    buffers, the step on device buffers, one D2H copy of the mask row.
    # The status word is sticky (first error kept) and is read once after each
    # run.  Each is replayed from CUDA graphs; the in-place one also eagerly.
    E = min(args.e2e_steps, K)
    rec = 528                                   # int16: 512 query + 2 position + 14 pad
    in_np = np.zeros((256, rec), np.int16)
    in_np[:, :512] = wl.q_host0.view(np.int16)
    in_np[:, 512:514] = np.arange(FIRST_POS, TOKENS, dtype=np.int32)[:, None].view(np.int16)
    in_host = torch.from_numpy(in_np).pin_memory()
    k_host = torch.from_numpy(np.ascontiguousarray(wl.keys_host0.view(np.int16))).pin_memory()
    mask_host = torch.empty((2, TOKENS), dtype=torch.uint8).pin_memory()
    in_dev = torch.empty(rec, dtype=torch.int16, device=device)

    def e2e_step(i):                            # in place
        k = steps[i]
        seq, j, p = wl.step_params(k)
        wl.step(k, q_src=in_host[j, :512].view(1, 512), pos_src=in_host[j, 512:514].view(torch.int32),
                keys_src=k_host, mask_dst=mask_host[i & 1])

    def e2e_step_copies(i):
        k = steps[i]
        seq, j, p = wl.step_params(k)
        in_dev.copy_(in_host[j], non_blocking=True)
        wl.keys[seq][p:p + 1].copy_(k_host[p:p + 1], non_blocking=True)
        wl.step(k, q_src=in_dev[:512].view(1, 512), pos_src=in_dev[512:514].view(torch.int32))
        mask_host[i & 1].copy_(wl.mask[seq][0], non_blocking=True)

    for fn in (e2e_step, e2e_step_copies):      # eager warm-up of both forms
        fn(0)
    torch.cuda.synchronize()
    e_graphs = capture_graphs(torch, e2e_step, list(range(E)))
    e2e_ms = time_graphs(torch, e_graphs)
    assert qsa.qsa_read_status(wl.status)[0] == 0
    c_graphs = capture_graphs(torch, e2e_step_copies, list(range(E)))
    copies_ms = time_graphs(torch, c_graphs)
    assert qsa.qsa_read_status(wl.status)[0] == 0
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e_start.record()
    for i in range(E):
        e2e_step(i)
    e_end.record()
    torch.cuda.synchronize()
    eager_ms = e_start.elapsed_time(e_end)
    assert qsa.qsa_read_status(wl.status)[0] == 0
    # bytes crossing the link per step: the record's query row and position,
    # one block's four raw keys every fourth step, the mask row
    e2e = {"value": world * E / (e2e_ms / 1000.0), "unit": "rows/s",
           "h2d_bytes_per_step": 512 * 2 + 4 + 128 * 2, "d2h_bytes_per_step": TOKENS,
           "steps": E,
           "path": "qsa_decode_index_select with inputs and mask row in pinned host memory, "
                   "read and written in place by the kernels, replayed from CUDA graphs",
           "eager_value": world * E / (eager_ms / 1000.0),
           "copies_value": world * E / (copies_ms / 1000.0),
           "copies_path": "the same steps with 2 H2D + 1 D2H cudaMemcpyAsync per step into "
                          "device buffers, replayed from CUDA graphs"}

    secondary = {}
    if not args.no_secondary:
        secondary["prefill_2304"] = prefill_2304(torch, qsa, device, hbm_gbs, bf16_tf)
        secondary["select_256k"] = select_256k(torch, qsa, device, hbm_gbs)
        secondary["prefill_chunk_64k"] = prefill_chunk(torch, qsa, device, hbm_gbs, bf16_tf)
        secondary["decode_long_32seq"] = decode_long(torch, qsa, device, hbm_gbs)
        secondary["decode_gather_64k"] = decode_gather(torch, qsa, device, hbm_gbs)
        secondary["prefill_attn_64k"] = prefill_attn(torch, qsa, device, hbm_gbs, bf16_tf)
        secondary["qk_proj"] = qk_proj(torch, qsa, device, bf16_tf)

    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 math, u8 mask",
        "data": "synthetic (seeded N(0,1) bf16 keys and queries, per-token log-uniform key scale)",
        "config": {"workload": WORKLOAD, "tokens": TOKENS, "budget": BUDGET, "rows_per_step": 1,
                   "sequences_rotated": R, "bytes_per_sequence": per_seq_bytes,
                   "l2": "inputs larger than L2 (steps rotate over the sequences)",
                   "launch": "CUDA graphs of 256 steps; per step qsa_decode_index_select: "
                             "one fused launch (pool the completed block, score, select)",
                   "pool_steps_timed": pool_steps_timed,
                   "step_schedule": "step k: sequence k mod R, position 65280 + k mod 256; "
                                    "a step whose token completes a block pools it",
                   "parallelism": f"replicas x{world}"},
        "three_entry_points_us_per_step": three_us,
        "roofline": roofline, "kernels": kernels, "clocks": clk, "e2e": e2e,
        "gpu_launches": int(K),  # one fused launch per step (it pools the new block itself)
        "secondary": secondary,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        for name in ("prefill_2304", "prefill_chunk_64k", "decode_long_32seq", "select_256k"):
            if name in secondary:
                secondary[name]["oracle_single_thread"] = oracle_single_thread(name)
        rate, cores, rows, dt = oracle_decode_rate(args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle",
                                "sample": f"{rows} decode rows (pos 65280.., 64k ctx) in "
                                          f"{dt:.1f} s on {cores} host threads"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def select_256k(torch, qsa, device, hbm_gbs, ncu=False):
    """Selection at 256k: 1024 rows at p = 262143 (65536 blocks) with relu-sum-like
    scores (70% zeros, 64 levels), budget 2048; amortised over the rows, and one
    row at a time (rotating over the 1024 rows so inputs stay larger than L2)."""
    tokens, rows = 262144, 1024
    cols = tokens // 4
    rng = qi.rng_for(4)
    sc = torch.from_numpy(qi.stress_scores(rng, rows, cols)).to(device)
    pos = torch.full((rows,), tokens - 1, dtype=torch.int32, device=device)
    mask = torch.empty((rows, tokens), dtype=torch.uint8, device=device)
    st = qsa.new_status(device)
    for _ in range(2 if ncu else 3):
        qsa.qsa_select_mask(sc, cols, pos, rows, tokens, BUDGET, mask, st)
    torch.cuda.synchronize()
    if ncu:
        return None
    g = capture_graphs(torch, lambda k: qsa.qsa_select_mask(sc, cols, pos, rows, tokens, BUDGET,
                                                            mask, st), list(range(10)), chunk=10)
    ms = time_graphs(torch, g) / 10
    byts = rows * (cols * 4 + tokens)
    one = capture_graphs(torch, lambda k: qsa.qsa_select_mask(sc[k % rows:k % rows + 1], cols,
                                                              pos[:1], 1, tokens, BUDGET,
                                                              mask[k % rows:k % rows + 1], st),
                         list(range(512)), chunk=256)
    ms1 = time_graphs(torch, one) / 512
    code, _ = qsa.qsa_read_status(st)
    assert code == 0
    return {"rows": rows, "us_per_row_amortised": ms * 1000.0 / rows, "launch_us": ms * 1000.0,
            "achieved_gbs": byts / (ms * 1e-3) / 1e9, "frac_of_measured_hbm": byts / (ms * 1e-3) / 1e9 / hbm_gbs,
            "us_single_row": ms1 * 1000.0, "budget": BUDGET,
            "context": "pages' L20 radix select: 298 us/row at 256k (context only)"}


# ------------------------------------------------- oracle beside the GPU lines

def oracle_single_thread(kind: str):
    """The oracle, single-threaded, on a stated subset of a secondary workload:
    the same shapes and input distributions, drawn on the host by the seeded
    generators (the oracle never reads a buffer the GPU path wrote).  Returns
    {"us_per_row", "sample"}: a baseline printed beside the GPU figures, not a
    target."""
    import oracle

    orc = oracle.Oracle()
    clock = time.perf_counter
    if kind in ("prefill_2304", "prefill_chunk_64k"):
        if kind == "prefill_2304":
            T, first, n_rows, sample = 2304, 0, 2304, 64
        else:
            T, first, n_rows, sample = 65536, 61440, 4096, 64
        rng = qi.rng_for(0 if kind == "prefill_2304" else 2)
        qw, kw = qi.norm_weights(rng)
        raw = qi.raw_keys(rng, T)
        q = np.ascontiguousarray(qi.fused_qk(rng, sample)[:, :512])
        c, s = orc.rope_table(T, THETA)
        cache = np.zeros((T // 4, 128), np.uint16)
        if first:
            orc.pool_blocks(raw, 128, 0, first // 4, kw, c, s, EPS, block_keys=cache)
        t0 = clock()
        orc.pool_blocks(raw[first:], 128, first // 4, (T - first) // 4, kw, c, s, EPS,
                        block_keys=cache)
        t_pool = clock() - t0
        rows = np.linspace(first, T - 1, sample).astype(np.int32)
        sc = np.zeros((1, T // 4), np.float32)
        t0 = clock()
        for i, p in enumerate(rows):
            orc.score_rows(q[i:i + 1], 512, rows[i:i + 1], 1, T, qw, c, s, EPS, cache, sc, T // 4)
            orc.select_row(sc[0, :max(1, (p + 1) // 4)], int(p), T, BUDGET)
        t_rows = clock() - t0
        us = (t_pool / n_rows + t_rows / sample) * 1e6
        what = (f"pool of the {(T - first) // 4} new blocks amortised over {n_rows} rows, plus "
                f"score + select of {sample} rows spread evenly over positions {first}..{T - 1}")
    elif kind == "decode_long_32seq":
        rng = qi.rng_for(3)
        lens = qi.long_context_lengths(rng, 32)[:2]
        qw, kw = qi.norm_weights(rng)
        tokens = 262144
        c, s = orc.rope_table(tokens, THETA)
        t_rows = 0.0
        for i, L in enumerate(lens):
            rr = qi.rng_for(3, salt=i + 1)
            raw = qi.raw_keys(rr, int(L))
            q = np.ascontiguousarray(qi.fused_qk(rr, 1)[:, :512])
            cache = orc.pool_blocks(raw, 128, 0, int(L) // 4, kw, c, s, EPS)
            sc = np.zeros((1, int(L) // 4), np.float32)
            t0 = clock()
            orc.score_rows(q, 512, np.array([L - 1], np.int32), 1, tokens, qw, c, s, EPS, cache,
                           sc, int(L) // 4)
            orc.select_row(sc[0], int(L - 1), tokens, BUDGET)
            t_rows += clock() - t0
        us = t_rows / len(lens) * 1e6
        what = (f"score + select of {len(lens)} rows at lengths "
                f"{', '.join(str(int(x)) for x in lens)}")
    elif kind == "select_256k":
        tokens, sample = 262144, 16
        sc = qi.stress_scores(qi.rng_for(4), sample, tokens // 4)
        t0 = clock()
        for i in range(sample):
            orc.select_row(sc[i], tokens - 1, tokens, BUDGET)
        us = (clock() - t0) / sample * 1e6
        what = f"select of {sample} stress rows at p = 262143, budget {BUDGET}"
    else:
        raise ValueError(kind)
    return {"us_per_row": us, "rows_per_s": 1e6 / us, "cores": 1, "kind": "oracle",
            "sample": what}


def prefill_2304(torch, qsa, device, hbm_gbs, bf16_tf, ncu=False):
    """Single-sequence prefill: T = 2304 tokens, every one of its 2304 rows
    queried, budget 2048 (rows up to p = 2050 keep their whole prefix, later
    rows truncate).  One step through qsa_index_select: pool the 576 blocks,
    score on the tensor cores, select; each stage also timed alone."""
    T = 2304
    nb = T // 4
    rng = qi.rng_for(0)
    fq_h = qi.fused_qk(rng, T)
    qw, kw = qi.norm_weights(rng)
    c, s = qsa.qsa_rope_tables(T, THETA)
    cd, sd = dev_tensor(torch, c, device), dev_tensor(torch, s, device)
    qw, kw = dev_tensor(torch, qw, device), dev_tensor(torch, kw, device)
    fq = dev_tensor(torch, fq_h, device)
    keys = fq.view(-1)[512:]
    pos = torch.arange(T, dtype=torch.int32, device=device)
    cache = torch.zeros((nb, 128), dtype=torch.int16, device=device)
    cols = nb
    sc = torch.empty((T, cols), dtype=torch.float32, device=device)
    mask = torch.empty((T, T), dtype=torch.uint8, device=device)
    st = qsa.new_status(device)
    ws = qsa.new_workspace(T, device)

    def fused():
        qsa.qsa_index_select(keys, 640, 0, nb, kw, fq, 640, pos, T, T, qw, cd, sd, T, EPS, BUDGET,
                             cache, sc, cols, mask, st, workspace=ws)

    def pool():
        qsa.qsa_pool_blocks(keys, 640, 0, nb, kw, cd, sd, T, EPS, cache)

    def score():
        qsa.qsa_score_rows(fq, 640, pos, None, T, T, qw, cd, sd, T, EPS, cache, None, sc, cols, st,
                           workspace=ws)

    def select():
        qsa.qsa_select_mask(sc, cols, pos, T, T, BUDGET, mask, st)

    for _ in range(2 if ncu else 3):
        fused()
    torch.cuda.synchronize()
    if ncu:
        return None
    it = 20
    t_fused = time_fn(torch, fused, it)
    t_pool = time_fn(torch, pool, it)
    t_score = time_fn(torch, score, it)
    t_sel = time_fn(torch, select, it)
    code, row = qsa.qsa_read_status(st)
    assert code == 0, (code, row)
    live = sum((p + 1) // 4 for p in range(T))
    trunc = sum((p + 1) // 4 for p in range(T) if (p + 1) // 4 > BUDGET // 4)
    flops = 1024.0 * live
    sel_bytes = 4.0 * trunc + T * T
    return {
        "rows": T, "tokens": T, "budget": BUDGET,
        "first_truncating_row": next(p for p in range(T) if (p + 1) // 4 > BUDGET // 4),
        "rows_per_s": T / (t_fused * 1e-3), "us_per_row": t_fused * 1000.0 / T,
        "step_us": t_fused * 1000.0,
        "path": "qsa_index_select (pool 576 blocks, tcgen05 score, select), CUDA graph",
        "pool": {"us": t_pool * 1000.0, "blocks": nb,
                 "frac_of_measured_hbm": nb * POOL_BYTES_PER_BLOCK / (t_pool * 1e-3) / 1e9 / hbm_gbs},
        "score_tcgen05": {"us": t_score * 1000.0, "live_scores": live,
                          "achieved_tflops": flops / (t_score * 1e-3) / 1e12,
                          "frac_of_measured_bf16": flops / (t_score * 1e-3) / 1e12 / bf16_tf},
        "select": {"us": t_sel * 1000.0, "algorithmic_bytes": sel_bytes,
                   "frac_of_measured_hbm": sel_bytes / (t_sel * 1e-3) / 1e9 / hbm_gbs},
        "note": "latency-bound: 0.68 GFLOP and 5.3 MB of mask, a few microseconds of work "
                "at either peak",
    }


def time_fn(torch, fn, iters):
    g = capture_graphs(torch, lambda k: fn(), list(range(iters)), chunk=iters)
    return time_graphs(torch, g) / iters


def prefill_chunk(torch, qsa, device, hbm_gbs, bf16_tf, ncu=False):
    """Chunked prefill: a 4096-row chunk at positions 61440..65535 of a 64k
    sequence.  Pool the chunk's 1024 new blocks, score 4096 rows on the tensor
    cores ([16384, 128] x [128, 16384] with the relu / head-sum epilogue), select."""
    tokens, first, rows = 65536, 61440, 4096
    nb = tokens // 4
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    cd, sd = dev_tensor(torch, c, device), dev_tensor(torch, s, device)
    rng = qi.rng_for(2)
    qw, kw = qi.norm_weights(rng)
    qw, kw = dev_tensor(torch, qw, device), dev_tensor(torch, kw, device)
    raw = qi.torch_normal_bf16(torch, (tokens, 128), qi.seed_for(2, 1), device)
    fq = qi.torch_normal_bf16(torch, (rows, 640), qi.seed_for(2, 2), device)
    cache = torch.zeros((nb, 128), dtype=torch.int16, device=device)
    qsa.qsa_pool_blocks(raw.view(-1), 128, 0, first // 4, kw, cd, sd, tokens, EPS, cache)
    pos = torch.arange(first, tokens, dtype=torch.int32, device=device)
    sc = torch.empty((rows, nb), dtype=torch.float32, device=device)
    mask = torch.empty((rows, tokens), dtype=torch.uint8, device=device)
    st = qsa.new_status(device)

    def pool():
        qsa.qsa_pool_blocks(raw[first:].reshape(-1), 128, first // 4, 1024, kw, cd, sd, tokens,
                            EPS, cache)

    def pool_all():  # the whole 64k sequence's 16384 blocks (rewrites the same keys)
        qsa.qsa_pool_blocks(raw.view(-1), 128, 0, nb, kw, cd, sd, tokens, EPS, cache)

    ws = qsa.new_workspace(rows, device)

    def score():
        qsa.qsa_score_rows(fq, 640, pos, None, rows, tokens, qw, cd, sd, tokens, EPS, cache, None,
                           sc, nb, st, workspace=ws)

    def select():
        qsa.qsa_select_mask(sc, nb, pos, rows, tokens, BUDGET, mask, st)

    def step():
        pool()
        score()
        select()

    def fused():  # the same step through the fused entry, qsa_index_select
        qsa.qsa_index_select(raw[first:].reshape(-1), 128, first // 4, 1024, kw, fq, 640, pos, rows,
                             tokens, qw, cd, sd, tokens, EPS, BUDGET, cache, sc, nb, mask, st,
                             workspace=ws)

    for _ in range(2 if ncu else 3):
        step()
        fused()
    torch.cuda.synchronize()
    if ncu:
        return None
    it = 10
    t_step = time_fn(torch, step, it)
    t_fused = time_fn(torch, fused, it)
    t_pool = time_fn(torch, pool, it)
    t_pool_all = time_fn(torch, pool_all, it)
    t_score = time_fn(torch, score, it)
    t_sel = time_fn(torch, select, it)
    code, row = qsa.qsa_read_status(st)
    assert code == 0, (code, row)
    live = int(sum((p + 1) // 4 for p in range(first, tokens)))
    flops = 1024.0 * live
    score_bytes = 4.0 * live + nb * 256 + rows * 512 * 2
    sel_bytes = 4.0 * live + rows * tokens
    pool_bytes = 1024 * POOL_BYTES_PER_BLOCK
    return {
        "rows": rows, "rows_per_s": rows / (t_step * 1e-3), "step_us": t_step * 1000.0,
        "fused_index_select_us": t_fused * 1000.0,
        "fused_rows_per_s": rows / (t_fused * 1e-3),
        "pool": {"us": t_pool * 1000.0, "blocks": 1024,
                 "frac_of_measured_hbm": pool_bytes / (t_pool * 1e-3) / 1e9 / hbm_gbs},
        "pool_all_16384": {"us": t_pool_all * 1000.0, "blocks": nb,
                           "frac_of_measured_hbm": nb * POOL_BYTES_PER_BLOCK / (t_pool_all * 1e-3)
                           / 1e9 / hbm_gbs},
        "score_tcgen05": {"us": t_score * 1000.0, "live_scores": live,
                          "achieved_tflops": flops / (t_score * 1e-3) / 1e12,
                          "frac_of_measured_bf16": flops / (t_score * 1e-3) / 1e12 / bf16_tf,
                          "achieved_gbs": score_bytes / (t_score * 1e-3) / 1e9,
                          "frac_of_measured_hbm": score_bytes / (t_score * 1e-3) / 1e9 / hbm_gbs},
        "select": {"us": t_sel * 1000.0, "achieved_gbs": sel_bytes / (t_sel * 1e-3) / 1e9,
                   "frac_of_measured_hbm": sel_bytes / (t_sel * 1e-3) / 1e9 / hbm_gbs},
    }


def decode_long(torch, qsa, device, hbm_gbs, ncu=False):
    """Decode at long context: 32 sequences, one row each, lengths U[131072, 262144],
    per-sequence key caches addressed by key_base, score_cols 65536, tokens 262144.
    Also times pooling every complete block of all 32 sequences (the pool
    throughput case)."""
    n_seq, tokens = 32, 262144
    rng = qi.rng_for(3)
    lens = qi.long_context_lengths(rng, n_seq)
    nbs = lens // 4
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    cd, sd = dev_tensor(torch, c, device), dev_tensor(torch, s, device)
    qw, kw = qi.norm_weights(rng)
    qw, kw = dev_tensor(torch, qw, device), dev_tensor(torch, kw, device)
    tok_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    blk_off = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int64)
    raw = qi.torch_normal_bf16(torch, (int(tok_off[-1]), 128), qi.seed_for(3, 1), device)
    cache = torch.zeros((int(blk_off[-1]) + 8, 128), dtype=torch.int16, device=device)

    def pool_all():
        for i in range(n_seq):
            qsa.qsa_pool_blocks(raw[tok_off[i]:tok_off[i + 1]].reshape(-1), 128, 0, int(nbs[i]),
                                kw, cd, sd, tokens, EPS, cache[blk_off[i]:])

    pool_all()
    q = qi.torch_normal_bf16(torch, (n_seq, 512), qi.seed_for(3, 2), device)
    pos = torch.from_numpy((lens - 1).astype(np.int32)).to(device)
    base = torch.from_numpy(blk_off[:-1].copy()).to(device)
    cols = 65536
    sc = torch.empty((n_seq, cols), dtype=torch.float32, device=device)
    mask = torch.empty((n_seq, tokens), dtype=torch.uint8, device=device)
    st = qsa.new_status(device)

    def score():
        qsa.qsa_score_rows(q, 512, pos, None, n_seq, tokens, qw, cd, sd, tokens, EPS, cache, base,
                           sc, cols, st)

    def select():
        qsa.qsa_select_mask(sc, cols, pos, n_seq, tokens, BUDGET, mask, st)

    for _ in range(2 if ncu else 3):
        score()
        select()
    torch.cuda.synchronize()
    if ncu:
        return None
    t_pool = time_fn(torch, pool_all, 3)
    t_score = time_fn(torch, score, 10)
    t_sel = time_fn(torch, select, 10)
    code, row = qsa.qsa_read_status(st)
    assert code == 0, (code, row)
    blocks = int(nbs.sum())
    sb = SCORE_BYTES_PER_BLOCK * blocks
    selb = 4 * blocks + n_seq * tokens
    pb = POOL_BYTES_PER_BLOCK * blocks
    return {
        "sequences": n_seq, "blocks": blocks, "rows_per_s": n_seq / ((t_score + t_sel) * 1e-3),
        "score": {"us": t_score * 1000.0, "achieved_gbs": sb / (t_score * 1e-3) / 1e9,
                  "frac_of_measured_hbm": sb / (t_score * 1e-3) / 1e9 / hbm_gbs},
        "select": {"us": t_sel * 1000.0, "achieved_gbs": selb / (t_sel * 1e-3) / 1e9,
                   "frac_of_measured_hbm": selb / (t_sel * 1e-3) / 1e9 / hbm_gbs},
        "pool_all_blocks": {"us": t_pool * 1000.0, "launches": n_seq,
                            "achieved_gbs": pb / (t_pool * 1e-3) / 1e9,
                            "frac_of_measured_hbm": pb / (t_pool * 1e-3) / 1e9 / hbm_gbs},
    }


def decode_gather(torch, qsa, device, hbm_gbs, ncu=False, rows=64):
    """The decode chain after selection at 64k: 64 sequences, one row each at
    p = 65534 (2051 selected tokens: 512 kept blocks and the 3-token tail),
    each with its own paged K/V cache (pages of 16 tokens, 2 KV heads x 256
    bf16, the pages of a sequence shuffled over the pool).  Times the token
    lists of all 64 mask rows, the gather of their K/V rows, and one row's
    list + gather (rotating over the 64 rows so each call reads cold data)."""
    tokens = TOKENS
    cols = tokens // 4
    g = torch.Generator(device=device)
    g.manual_seed(qi.seed_for(5))
    sc = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    pos = torch.full((rows,), tokens - 2, dtype=torch.int32, device=device)
    mask = torch.empty((rows, tokens), dtype=torch.uint8, device=device)
    st = qsa.new_status(device)
    qsa.qsa_select_mask(sc, cols, pos, rows, tokens, BUDGET, mask, st)
    table_len = tokens // GATHER_PAGE
    pages = rows * table_len
    k_pool = torch.randint(-32768, 32767, (pages * GATHER_PAGE, GATHER_WIDTH), generator=g,
                           device=device, dtype=torch.int16)
    v_pool = torch.randint(-32768, 32767, (pages * GATHER_PAGE, GATHER_WIDTH), generator=g,
                           device=device, dtype=torch.int16)
    perm = torch.stack([torch.randperm(table_len, generator=g, device=device)
                        for _ in range(rows)])
    table = (perm + torch.arange(rows, device=device)[:, None] * table_len).to(torch.int32)
    sel_cols = BUDGET + 3
    sel = torch.empty((rows, sel_cols), dtype=torch.int32, device=device)
    n_sel = torch.zeros(rows, dtype=torch.int32, device=device)
    k_out = torch.empty((rows * sel_cols, GATHER_WIDTH), dtype=torch.int16, device=device)
    v_out = torch.empty_like(k_out)

    def tokens_all():
        qsa.qsa_mask_tokens(mask, rows, tokens, sel, sel_cols, n_sel)

    def gather_all():
        qsa.qsa_gather_kv(k_pool, v_pool, GATHER_WIDTH, pages, table, table_len, table_len,
                          GATHER_PAGE, sel, sel_cols, n_sel, rows, sel_cols, k_out, v_out,
                          sel_cols, st)

    def one_row(k):
        r = k % rows
        qsa.qsa_mask_tokens(mask[r], 1, tokens, sel[r], sel_cols, n_sel[r:r + 1])
        qsa.qsa_gather_kv(k_pool, v_pool, GATHER_WIDTH, pages, table[r], table_len, table_len,
                          GATHER_PAGE, sel[r], sel_cols, n_sel[r:r + 1], 1, sel_cols,
                          k_out[r * sel_cols:], v_out[r * sel_cols:], sel_cols, st)

    for _ in range(2 if ncu else 3):
        tokens_all()
        gather_all()
    torch.cuda.synchronize()
    if ncu:
        return None
    t_tok = time_fn(torch, tokens_all, 10)
    t_gat = time_fn(torch, gather_all, 10)
    gr = capture_graphs(torch, one_row, list(range(256)), chunk=256)
    t_one = time_graphs(torch, gr) / 256
    code, row = qsa.qsa_read_status(st)
    assert code == 0, (code, row)
    n = int(n_sel.sum())
    tb = rows * tokens + 4 * n + 4 * rows
    gb = GATHER_BYTES_PER_TOKEN * n
    return {
        "rows": rows, "selected_tokens": n, "width": GATHER_WIDTH, "page_size": GATHER_PAGE,
        "mask_tokens": {"us": t_tok * 1000.0, "achieved_gbs": tb / (t_tok * 1e-3) / 1e9,
                        "frac_of_measured_hbm": tb / (t_tok * 1e-3) / 1e9 / hbm_gbs},
        "gather_kv": {"us": t_gat * 1000.0, "achieved_gbs": gb / (t_gat * 1e-3) / 1e9,
                      "frac_of_measured_hbm": gb / (t_gat * 1e-3) / 1e9 / hbm_gbs},
        "one_row_list_and_gather_us": t_one * 1000.0,
    }


def prefill_attn(torch, qsa, device, hbm_gbs, bf16_tf, ncu=False, rows=4096):
    """Sparse prefill attention on the chunked-prefill shape: rows at positions
    65536 - rows .. 65535 of one 64k sequence, each attending its 2048 selected
    tokens plus tail (lists from the device selection of random scores), 16
    query heads over 2 KV heads of 256, pages of 16 shuffled over the pool."""
    tokens, first = TOKENS, TOKENS - rows
    nq, nkv, hd, page = 16, 2, 256, 16
    cols = tokens // 4
    g = torch.Generator(device=device)
    g.manual_seed(qi.seed_for(7))
    sc = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    pos = torch.arange(first, tokens, dtype=torch.int32, device=device)
    mask = torch.empty((rows, tokens), dtype=torch.uint8, device=device)
    st = qsa.new_status(device)
    qsa.qsa_select_mask(sc, cols, pos, rows, tokens, BUDGET, mask, st)
    sel_cols = BUDGET + 3
    sel = torch.empty((rows, sel_cols), dtype=torch.int32, device=device)
    n_sel = torch.zeros(rows, dtype=torch.int32, device=device)
    qsa.qsa_mask_tokens(mask, rows, tokens, sel, sel_cols, n_sel)
    del sc, mask
    table_len = tokens // page
    kv_shape = (table_len * page, nkv * hd)
    k_pool = (torch.randn(kv_shape, generator=g, device=device) * 1.0).to(torch.bfloat16).view(torch.int16)
    v_pool = (torch.randn(kv_shape, generator=g, device=device) * 1.0).to(torch.bfloat16).view(torch.int16)
    table = torch.randperm(table_len, generator=g, device=device).to(torch.int32)
    q = (torch.randn((rows, nq * hd), generator=g, device=device) * 2.0).to(torch.bfloat16).view(torch.int16)
    out = torch.empty((rows, nq * hd), dtype=torch.int16, device=device)

    def attn():
        qsa.qsa_sparse_attn(q, nq * hd, nq, nkv, hd, k_pool, v_pool, table_len, page, table,
                            table_len, 0, sel, sel_cols, n_sel, rows, sel_cols, 1.0 / 16.0, out,
                            nq * hd, st)

    for _ in range(2 if ncu else 3):
        attn()
    torch.cuda.synchronize()
    if ncu:
        return None
    t = time_fn(torch, attn, 10)
    code, row = qsa.qsa_read_status(st)
    assert code == 0, (code, row)
    n = int(n_sel.sum())
    gathered = n * nkv * hd * 2 * 2 + rows * nq * hd * 2 * 2 + n * 4
    unique = 2 * kv_shape[0] * kv_shape[1] * 2 + rows * nq * hd * 2 * 2 + n * 4
    flops = 4.0 * nq * hd * n
    return {
        "rows": rows, "selected_tokens": n, "heads": f"{nq}q/{nkv}kv x {hd}", "page_size": page,
        "us": t * 1000.0, "rows_per_s": rows / (t * 1e-3),
        "gathered_gbs": gathered / (t * 1e-3) / 1e9,
        "unique_bytes": unique, "unique_frac_of_measured_hbm": unique / (t * 1e-3) / 1e9 / hbm_gbs,
        "achieved_tflops": flops / (t * 1e-3) / 1e12,
        "frac_of_measured_bf16": flops / (t * 1e-3) / 1e12 / bf16_tf,
    }


def qk_proj(torch, qsa, device, bf16_tf, ncu=False):
    """The indexer's qk projection on tcgen05: one 2048-row slab (the pages'
    slab) and a 4096-row prefill chunk, hidden 2560 -> 640, bf16."""
    hidden, out_cols = 2560, 640
    g = torch.Generator(device=device)
    g.manual_seed(qi.seed_for(9))
    w = (torch.randn((out_cols, hidden), generator=g, device=device) * 0.02).to(torch.bfloat16).view(torch.int16)
    st = qsa.new_status(device)
    res = {"hidden": hidden, "out_cols": out_cols}
    for rows in (2048, 4096):
        x = torch.randn((rows, hidden), generator=g, device=device).to(torch.bfloat16).view(torch.int16)
        y = torch.empty((rows, out_cols), dtype=torch.int16, device=device)

        def proj():
            qsa.qsa_qk_proj(x, hidden, w, rows, hidden, out_cols, y, out_cols, st)

        for _ in range(2 if ncu else 3):
            proj()
        torch.cuda.synchronize()
        if ncu:
            continue
        t = time_fn(torch, proj, 20)
        flops = 2.0 * rows * hidden * out_cols
        res[f"rows_{rows}"] = {"us": t * 1000.0, "achieved_tflops": flops / (t * 1e-3) / 1e12,
                               "frac_of_measured_bf16": flops / (t * 1e-3) / 1e12 / bf16_tf}
    code, row = qsa.qsa_read_status(st)
    assert code == 0, (code, row)
    return None if ncu else res


# ------------------------------------------------------------ ncu cases

def ncu_case(name: str):
    """Small eager cases for ncu captures: a few launches of each kernel, no
    timing, no graphs."""
    import torch

    import sparse_attention_token_qsa_gb300 as qsa

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    if name == "decode":
        wl = DecodeWorkload(torch, qsa, dev, 4)
        for k in range(8):
            wl.step(k)
    elif name == "prefill":
        prefill_chunk(torch, qsa, dev, 6800.0, 1900.0, ncu=True)
    elif name == "prefill2304":
        prefill_2304(torch, qsa, dev, 6800.0, 1900.0, ncu=True)
    elif name == "select256k":
        select_256k(torch, qsa, dev, 6800.0, ncu=True)
    elif name == "decode_long":
        decode_long(torch, qsa, dev, 6800.0, ncu=True)
    elif name == "gather":
        decode_gather(torch, qsa, dev, 6800.0, ncu=True)
    elif name == "proj":
        qk_proj(torch, qsa, dev, 1900.0, ncu=True)
    elif name == "attn":
        prefill_attn(torch, qsa, dev, 6800.0, 1900.0, ncu=True, rows=512)
    elif name == "gather_small":      # 8 rows: 1.1 GB of K/V pools
        decode_gather(torch, qsa, dev, 6800.0, ncu=True, rows=8)
    else:
        raise SystemExit(f"unknown ncu case {name}")
    torch.cuda.synchronize()
    print("ncu case done:", name)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group("gloo")
        run_reference(args, rank, world)
        return
    import torch

    if args.ncu_case:
        ncu_case(args.ncu_case)
        return
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    run_ours(args, rank, world, device)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
