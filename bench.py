#!/usr/bin/env python3
"""Benchmark of the fused attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill attention forward (attn_fwd) on the largest single-GPU prefill
    workload, long-context MHA causal B=1, H=32, N_q=N_kv=16384, d=128 with 1 %
    of the key rows scaled by 8 (the headline metric, TFLOP/s), and
  * MLA decode (mla_decode) on B=64, H=128, N_kv=4096, d_c=512, d_r=64
    (HBM GB/s, reported in the "decode" object).
The other prefill workloads (MHA causal B=4 H=16 N=2048, GQA 8k causal, its
causal and symmetric 256-key windows) are timed kernel-only as extra keys.

Timing: W untimed warm-up steps, then K timed steps.  Inputs are resident in
HBM; between steps a 256 MiB buffer (> the 129 MB L2) is overwritten so no
step starts with its inputs in L2.  Each kernel call is bracketed by CUDA
events on the launching stream (torch's current stream, which the binding
passes to the library); the flush is outside the brackets.  The run is
bracketed by a barrier + device synchronize on both sides and the maximum over
ranks is taken.  FLOPs count 4*d per allowed (query, key) pair; bytes count
each decode input read once and each output written once.

--impl reference times the fp64 CPU oracle (the reference of this project)
on a bounded sample of the same workload and prints the same JSON line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from tiled_attention_flashattention_gb300 import workloads as wl  # noqa: E402

METRIC = "attn fwd TFLOP/s and MLA-decode HBM GB/s on 1 GB300, % of roofline"
PREFILL = "mha_causal_spiky_b1_h32_n16384_d128"
DECODE = "mla_decode_b64_h128_nkv4096"
FLUSH_BYTES = 256 << 20
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- workload arithmetic
def key_bounds(i, N_q: int, N_kv: int, causal: bool, window: int):
    """Inclusive visible-key bounds (lo, hi) of query rows i (int64 array)."""
    off = N_kv - N_q
    if causal:
        hi = np.minimum(N_kv - 1, i + off)
        lo = np.maximum(0, i + off - window + 1) if window > 0 else np.zeros_like(i)
    elif window > 0:        # symmetric local window
        hi = np.minimum(N_kv - 1, i + off + window)
        lo = np.maximum(0, i + off - window)
    else:
        hi, lo = np.full_like(i, N_kv - 1), np.zeros_like(i)
    return lo, hi


def allowed_pairs(N_q: int, N_kv: int, causal: bool, window: int) -> int:
    """Number of (query, key) pairs the mask keeps, per (batch, head)."""
    lo, hi = key_bounds(np.arange(N_q, dtype=np.int64), N_q, N_kv, causal, window)
    return int(np.maximum(0, hi - lo + 1).sum())


def prefill_form(c: wl.PrefillCase) -> str:
    """Which instance of the prefill kernel the library launches for this
    workload: the host picks two 128-row Q tiles per CTA (128-key tiles) when
    a query tile visits at least 16 128-key tiles on average, else one Q tile
    on 64-key tiles, pipelined (same rule as the launcher)."""
    lo, hi = key_bounds(np.arange(c.N_q, dtype=np.int64), c.N_q, c.N_kv, c.causal, c.window)
    tiles = []
    for t0 in range(0, c.N_q, 128):
        klo, khi = lo[t0:t0 + 128].min(), hi[t0:t0 + 128].max() + 1
        tiles.append(max(0, -(-khi // 128) - klo // 128) if khi > klo else 0)
    if np.mean(tiles) >= 16:
        return f"attn_fwd_kernel<{c.d}, dense, 2 Q tiles per CTA, 128-key tiles>"
    return f"attn_fwd_kernel<{c.d}, dense, 1 Q tile per CTA, 64-key tiles, pipelined>"


def bench_config(pc, dc, world):
    return {"workload": pc.name, "B": pc.B, "H": pc.H, "H_kv": pc.H_kv, "N_q": pc.N_q, "N_kv": pc.N_kv,
            "d": pc.d, "causal": pc.causal, "window": pc.window, "decode_workload": dc.name,
            "parallelism": f"independent shards x{world}" if world > 1 else "single GPU",
            "l2": "256 MiB buffer overwritten between steps (outside the timed kernels)"}


def prefill_flops(c: wl.PrefillCase) -> float:
    return 4.0 * c.d * allowed_pairs(c.N_q, c.N_kv, c.causal, c.window) * c.B * c.H


def prefill_bytes(c: wl.PrefillCase) -> float:
    return 2.0 * (c.B * c.H * c.N_q * c.d * 2 + c.B * c.H_kv * c.N_kv * c.d * 2) + 4.0 * c.B * c.H * c.N_q


def decode_flops(c: wl.MlaCase) -> float:
    return float(c.B * c.H * c.N_kv) * (2 * (c.d_c + c.d_r) + 2 * c.d_c)


def decode_bytes(c: wl.MlaCase) -> float:
    kv = c.B * c.N_kv * (c.d_c + c.d_r) * 2
    q = c.B * c.H * (c.d_c + c.d_r) * 2
    out = c.B * c.H * c.d_c * 2 + c.B * c.H * 4
    return float(kv + q + out)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


def kernel_source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in ("ptx.cuh",) + names:
        with open(os.path.join(ROOT, "tiled_attention_flashattention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch(kernel_key: str, source: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, or
    None when the summary is missing or the kernel source changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            d = json.load(f)[kernel_key]
    except (OSError, KeyError, ValueError):
        return None
    if d.get("source_hash") != kernel_source_hash(source) or d.get("workload") != workload:
        return None
    return d.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi polled every 20 ms in a child process (read-only queries).
    start() returns once the first sample has been written, so that a short
    timed region that follows is covered; summary(t0, t1) reports the samples
    from wall time t0 to t1 (time.time())."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.rows = []
        self.path = os.path.join(tempfile.gettempdir(), f"gbattn_clocks_{os.getpid()}.csv")

    def start(self, wait_s: float = 5.0):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        t_end = time.time() + wait_s
        while time.time() < t_end:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    @staticmethod
    def _parse_time(stamp: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                continue
        return None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                self.rows.append((self._parse_time(parts[0]), float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue

    def summary(self, t0: float, t1: float, timed=None):
        """Samples taken from t0 to t1 (wall clock; nvidia-smi stamps local time).
        timed = (ta, tb): also count the samples inside the timed region."""
        rows = [r for r in self.rows if r[0] is not None and t0 - 0.05 <= r[0] <= t1 + 0.05]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({self.NAMES[k] for r in rows for k, v in enumerate(r[3]) if v == "Active"})
        out = {"sm_mhz": statistics.median(r[1] for r in rows), "sm_mhz_min": min(r[1] for r in rows),
               "sm_max_mhz": max(r[2] for r in rows), "reasons": reasons, "samples": len(rows),
               "window": "from the first timed step to the end of the extra workloads"}
        if timed:
            ta, tb = timed
            out["samples_in_timed_steps"] = sum(1 for r in rows if ta - 0.025 <= r[0] <= tb + 0.025)
        return out


# ---------------------------------------------------------------- distributed plumbing
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle timing (CPU)
def oracle_sample_rate(case, rows, kind):
    """Time the oracle on the given rows; returns (seconds, flops)."""
    import oracle
    t0 = time.perf_counter()
    if kind == "prefill":
        Q, K, V = case["inputs"]
        c = case["case"]
        oracle.attn_fwd(Q, K, V, c.causal, c.window, c.softmax_scale(), rows=rows)
        lo, hi = key_bounds(np.asarray(rows, dtype=np.int64) % c.N_q, c.N_q, c.N_kv, c.causal, c.window)
        flops = float((4 * c.d * np.maximum(0, hi - lo + 1)).sum())
    else:
        Qn, Qp, KV, Kp = case["inputs"]
        c = case["case"]
        oracle.mla_decode(Qn, Qp, KV, Kp, c.softmax_scale(), rows=rows)
        flops = float(len(rows) * c.N_kv * (2 * (c.d_c + c.d_r) + 2 * c.d_c))
    return time.perf_counter() - t0, flops


def cpu_baseline(pcase, dcase, budget_s: float):
    """Oracle on a bounded sample: every stride-th prefill row (stride chosen
    from a short calibration so the sample takes about budget_s)."""
    import oracle
    c = pcase["case"]
    total_rows = c.B * c.H * c.N_q
    cal_rows = np.arange(0, total_rows, max(1, total_rows // 512), dtype=np.int64)
    dt, fl = oracle_sample_rate(pcase, cal_rows, "prefill")
    rate = fl / max(dt, 1e-6)
    stride = max(1, int(math.ceil(prefill_flops(c) / (rate * budget_s))))
    rows = np.arange(0, total_rows, stride, dtype=np.int64)
    dt, fl = oracle_sample_rate(pcase, rows, "prefill")
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle on {len(rows)} of {total_rows} query rows (every {stride}th row) of "
                      f"{c.name}; {fl / 1e9:.1f} GFLOP in {dt:.1f} s"}


# ---------------------------------------------------------------- main arms
def run_reference(args, rank, world):
    if rank != 0:
        return
    pc = wl.WORKLOADS[args.workload]
    pcase = {"case": pc, "inputs": wl.prefill_inputs(pc)}
    import oracle
    total_rows = pc.B * pc.H * pc.N_q
    # size each step so that warm-up + timed steps take about 60 s of CPU time
    cal_rows = np.arange(0, total_rows, max(1, total_rows // 256), dtype=np.int64)
    dt, fl = oracle_sample_rate(pcase, cal_rows, "prefill")
    rate = fl / max(dt, 1e-6)
    per_step_s = max(0.05, 60.0 / (args.steps + args.warmup))
    stride = max(1, int(math.ceil(prefill_flops(pc) / (rate * per_step_s))))
    rows = np.arange(0, total_rows, stride, dtype=np.int64)
    for _ in range(args.warmup):
        oracle_sample_rate(pcase, rows, "prefill")
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = oracle_sample_rate(pcase, rows, "prefill")
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = (f"fp64 oracle, {len(rows)} of {total_rows} query rows (every {stride}th) of {pc.name} "
              f"per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": bench_config(pc, wl.WORKLOADS[args.decode_workload], world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.default_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def paged_inputs(dev, H=128, s_q=1):
    """64 sequences with seeded lengths in [2048, 6144] keys (mean about 4096),
    64-key pages placed at random, H heads and s_q query tokens per sequence."""
    g = torch.Generator().manual_seed(wl.SEED_BASE + 5)
    lens = torch.randint(2048, 6145, (64,), generator=g).tolist()
    xs = [x.to(dev) for x in wl.random_mla_paged(H, lens, seed=wl.SEED_BASE + 5, s_q=s_q)]
    return lens, xs


def paged_decode_workload(gb, dev, peaks, flush, reps=10, H=128, s_q=1):
    """Kernel-only HBM GB/s of mla_decode_paged on 64 sequences with seeded
    lengths in [2048, 6144] keys (mean about 4096) in 64-key pages placed at
    random (inputs resident, L2 flushed before each timed call).  With H heads
    and s_q query tokens per sequence; when s_q * H <= 128 all of a sequence's
    tokens share one 128-row tile and its keys are read once.  Algorithmic
    bytes: every key row read once (576 bf16), Q read once, O and LSE written
    once."""
    lens, (Qn, Qp, KV, Kp, table, L) = paged_inputs(dev, H, s_q)
    B = len(lens)
    lead = (B, s_q, H) if s_q > 1 else (B, H)
    O = torch.empty(*lead, 512, dtype=torch.bfloat16, device=dev)
    LSE = torch.empty(*lead, dtype=torch.float32, device=dev)
    ws = torch.empty(gb.mla_decode_paged_workspace_bytes(B, s_q, H), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(576)
    call = lambda: gb.mla_decode_paged(Qn, Qp, KV, Kp, table, L, scale=scale, O=O, LSE=LSE, workspace=ws)
    for _ in range(3):
        call()
    stream = torch.cuda.current_stream(dev)
    total = 0.0
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1) / 1e3
    gb.check()
    t = total / reps
    rows = B * s_q * H
    by = float(sum(lens) * 576 * 2 + rows * 576 * 2 + rows * 512 * 2 + rows * 4)
    gbs = by / t / 1e9
    name = "mla_paged_b64_h128_len2048to6144_page64" if (H, s_q) == (128, 1) else \
        f"mla_paged_b64_h{H}_sq{s_q}_len2048to6144_page64"
    return {"workload": name, "gbs": gbs, "frac_hbm_peak": gbs / peaks["hbm_gbs"],
            "ms": t * 1e3, "total_keys": int(sum(lens)), "algorithmic_bytes": by, "heads": H, "s_q": s_q}


def sparse_pairs(mask, N_q: int, N_kv: int, causal: bool, window: int, block: int = 128) -> int:
    """(query, key) pairs that both the element mask and the block mask keep,
    summed over (batch, head).  mask: uint8 [B,H,ceil(N_q/block),ceil(N_kv/block)]."""
    i = np.arange(N_q, dtype=np.int64)
    lo, hi = key_bounds(i, N_q, N_kv, causal, window)
    kb = np.arange(-(-N_kv // block), dtype=np.int64)
    k0 = kb * block
    k1 = np.minimum(k0 + block, N_kv) - 1
    # allowed keys of row i inside key block kb: |[lo_i, hi_i] ∩ [k0, k1]|
    per = np.maximum(0, np.minimum(hi[:, None], k1[None, :]) - np.maximum(lo[:, None], k0[None, :]) + 1)
    qb = -(-N_q // block)
    per = np.pad(per, ((0, qb * block - N_q), (0, 0)))
    block_pairs = per.reshape(qb, block, -1).sum(1)                # [QB, KB]
    m = mask.numpy().astype(np.int64)                              # [B,H,QB,KB]
    return int((m * block_pairs[None, None]).sum())


def sparse_prefill_workload(gb, dev, peaks, flush, reps=10):
    """Kernel-only TFLOP/s of attn_fwd_sparse on the 8k causal GQA inputs with a
    seeded 25 %-density block mask (L2 flushed before each timed launch).  The
    algorithmic work counts only pairs inside active blocks that the causal
    mask keeps."""
    c = wl.WORKLOADS["gqa_causal_b2_h32_hkv8_n8192_d128"]
    mask_h = wl.random_block_mask(c.B, c.H, c.N_q, c.N_kv, 0.25, seed=wl.SEED_BASE + 6)
    Q, K, V = (x.to(dev) for x in wl.prefill_inputs(c))
    mask = mask_h.to(dev)
    O = torch.empty_like(Q)
    L = torch.empty(c.B, c.H, c.N_q, dtype=torch.float32, device=dev)
    call = lambda: gb.attn_fwd_sparse(Q, K, V, mask, causal=True, scale=c.softmax_scale(), O=O, LSE=L)
    for _ in range(3):
        call()
    stream = torch.cuda.current_stream(dev)
    total = 0.0
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1) / 1e3
    gb.check()
    t = total / reps
    flops = 4.0 * c.d * sparse_pairs(mask_h, c.N_q, c.N_kv, True, 0)
    tf = flops / t / 1e12
    return {"workload": "gqa_causal_sparse25_b2_h32_hkv8_n8192_d128", "tflops": tf,
            "frac_bf16_peak": tf / peaks["bf16_tflops"], "ms": t * 1e3,
            "active_blocks": int(mask_h.sum()), "algorithmic_flops": flops}


def ssd_flops(c) -> float:
    """FLOPs of the chunked SSD scan (128-step chunks): per (chunk, head) the
    causal intra-chunk products C B^T and W x over the Q(Q+1)/2 pairs s <= t
    (2N and 2P FLOPs per pair), the entering-state product C S^T (2QPN) and the
    chunk's state contribution (2QPN); the ragged last chunk counts its own
    length."""
    Q, total = 128, 0.0
    for c0 in range(0, c.L, Q):
        q = min(Q, c.L - c0)
        total += q * (q + 1) * (c.N + c.P) + 4.0 * q * c.P * c.N
    return total * c.Bsz * c.H


def ssd_bytes(c) -> float:
    """Algorithmic bytes: x (bf16) read and y (fp32) written once, dt read once,
    B and C (bf16) read once per group."""
    return float(c.Bsz * c.L * (c.H * (2 * c.P + 4 * c.P + 4) + c.G * 2 * 2 * c.N))


def ssd_workload(gb, dev, peaks, flush, reps=10):
    """Kernel-only throughput of ssd_scan on the Mamba-2-sized workload, inputs
    resident, L2 flushed before each timed call, CUDA events around the call.
    At this size the HBM time floor (algorithmic bytes / copy bandwidth) is
    about twice the tensor floor (algorithmic FLOPs / bf16 peak), so the
    roofline is HBM."""
    c = wl.SSD_WORKLOAD
    x, dt, A, B, C, D = (t.to(dev) for t in wl.ssd_inputs(c))
    y = torch.empty(c.Bsz, c.L, c.H, c.P, dtype=torch.float32, device=dev)
    S = torch.empty(c.Bsz, c.H, c.P, c.N, dtype=torch.float32, device=dev)
    call = lambda: gb.ssd_scan(x, dt, A, B, C, D, y=y, final_state=S)
    for _ in range(3):
        call()
    stream = torch.cuda.current_stream(dev)
    total = 0.0
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1) / 1e3
    gb.check()
    t = total / reps
    by = ssd_bytes(c) + c.Bsz * c.H * c.P * c.N * 4
    gbs = by / t / 1e9
    tf = ssd_flops(c) / t / 1e12
    del x, y, S
    return {"workload": c.name, "bound": "hbm", "gbs": gbs, "frac_hbm_peak": gbs / peaks["hbm_gbs"],
            "tflops": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"], "ms": t * 1e3,
            "algorithmic_bytes": by, "algorithmic_flops": ssd_flops(c), "launches_per_call": 1}


def other_prefill_workloads(gb, dev, skip, peaks, flush, reps=10):
    """Kernel-only TFLOP/s of the other prefill workloads (inputs resident,
    L2 flushed before each timed launch, CUDA events around the launch)."""
    out = {}
    stream = torch.cuda.current_stream(dev)
    for name, c in wl.WORKLOADS.items():
        if not isinstance(c, wl.PrefillCase) or name == skip or c.N_q < 1024:
            continue
        Q, K, V = (x.to(dev) for x in wl.prefill_inputs(c))
        O = torch.empty_like(Q)
        L = torch.empty(c.B, c.H, c.N_q, dtype=torch.float32, device=dev)
        for _ in range(3):
            gb.attn_fwd(Q, K, V, causal=c.causal, window=c.window, scale=c.softmax_scale(), O=O, LSE=L)
        total = 0.0
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gb.attn_fwd(Q, K, V, causal=c.causal, window=c.window, scale=c.softmax_scale(), O=O, LSE=L)
            e1.record(stream)
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1) / 1e3
        gb.check()
        t = total / reps
        tf = prefill_flops(c) / t / 1e12
        gbs = prefill_bytes(c) / t / 1e9
        out[name] = {"tflops": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"], "ms": t * 1e3,
                     "gbs": gbs, "frac_hbm_peak": gbs / peaks["hbm_gbs"]}
        del Q, K, V, O, L
    return out


def peaks_now():
    return load_peaks()[0]


def copy_ceiling(dev, ins, outs, flush, reps=5):
    """Seconds per step to move the given pinned host tensors to the device and
    the given device-sized results back with plain cudaMemcpyAsync (inputs on
    one stream, results on another, as in the host-buffer entry points), median
    of reps, wall time bracketed by device synchronisation."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    d_in = [torch.empty(x.shape, dtype=x.dtype, device=dev) for x in ins]
    d_out = [torch.empty(x.shape, dtype=x.dtype, device=dev) for x in outs]
    ts = []
    for _ in range(reps + 1):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(s_in):
            for d, h in zip(d_in, ins):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            for h, d in zip(outs, d_out):
                h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()
        ts.append(time.perf_counter() - t0)
    del d_in, d_out
    return statistics.median(ts[1:])


def run_ours(args, rank, world, local):
    import tiled_attention_flashattention_gb300 as gb
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from tiled_attention_flashattention_gb300 import _build
    _build.build()
    gb.load_library()

    pc = wl.WORKLOADS[args.workload]
    dc = wl.WORKLOADS[args.decode_workload]
    # per-rank inputs: independent shards (weak scaling), seeded per rank
    pc_r = wl.PrefillCase(**{**pc.__dict__, "seed": pc.seed + 1000 * rank})
    dc_r = wl.MlaCase(**{**dc.__dict__, "seed": dc.seed + 1000 * rank})
    Qh, Kh, Vh = wl.prefill_inputs(pc_r)
    dec_h = wl.mla_inputs(dc_r)
    Q, K, V = (x.to(dev) for x in (Qh, Kh, Vh))
    Qn, Qp, KV, Kp = (x.to(dev) for x in dec_h)
    O = torch.empty_like(Q)
    LSE = torch.empty(pc.B, pc.H, pc.N_q, dtype=torch.float32, device=dev)
    Od = torch.empty(dc.B, dc.H, dc.d_c, dtype=torch.bfloat16, device=dev)
    Ld = torch.empty(dc.B, dc.H, dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, gb.mla_decode_workspace_bytes(dc.B, dc.H, dc.N_kv, dc.d_c)), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale_p, scale_d = pc.softmax_scale(), dc.softmax_scale()

    def step(events=None):
        flush.zero_()
        if events:
            events[0].record(stream)
        gb.attn_fwd(Q, K, V, causal=pc.causal, window=pc.window, scale=scale_p, O=O, LSE=LSE)
        if events:
            events[1].record(stream)
        gb.mla_decode(Qn, Qp, KV, Kp, scale=scale_d, O=Od, LSE=Ld, workspace=ws)
        if events:
            events[2].record(stream)

    sampler = ClockSampler(local)
    sampler.start()          # returns once nvidia-smi has written its first sample
    for _ in range(max(3, args.warmup)):
        step()
    gb.check()
    n_ev = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_ev)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(evs[k])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    t_wall1 = time.time()
    barrier(world)
    gb.check()
    t_pre = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3   # seconds
    t_dec = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    t_pre = max_over_ranks(t_pre, world)
    t_dec = max_over_ranks(t_dec, world)

    peaks, peak_src = load_peaks()
    fl_p = prefill_flops(pc)
    by_d = decode_bytes(dc)
    pre_launch_s = t_pre / args.steps
    dec_launch_s = t_dec / args.steps
    tflops = fl_p * args.steps * world / t_pre / 1e12
    gbs = by_d * args.steps * world / t_dec / 1e9
    n_dec_launches = 2 if gb.mla_decode_workspace_bytes(dc.B, dc.H, dc.N_kv, dc.d_c) > 0 else 1

    # ---- end to end through the C ABI with host buffers: pinned host inputs in,
    # host results out; the library pipelines the copies with the kernels
    e2e_steps = max(3, min(args.steps, 20))
    Qh_p, Kh_p, Vh_p = (x.pin_memory() for x in (Qh, Kh, Vh))
    dec_p = [x.pin_memory() for x in dec_h]
    O_h = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    L_h = torch.empty(LSE.shape, dtype=LSE.dtype).pin_memory()
    Od_h = torch.empty(Od.shape, dtype=Od.dtype).pin_memory()
    Ld_h = torch.empty(Ld.shape, dtype=Ld.dtype).pin_memory()
    buf_p = torch.empty(gb.attn_fwd_host_device_bytes(pc.B, pc.H, pc.H_kv, pc.N_q, pc.N_kv, pc.d), dtype=torch.uint8,
                        device=dev)
    buf_d = torch.empty(gb.mla_decode_host_device_bytes(dc.B, dc.H, dc.N_kv, dc.d_c, dc.d_r), dtype=torch.uint8,
                        device=dev)
    e2e_pre, e2e_dec = 0.0, 0.0
    e2e_warm = max(3, args.warmup)      # the first calls also settle the host pipeline
    pre_ms = []                          # per-step prefill e2e times (ms), for the spread
    for k in range(e2e_steps + e2e_warm):
        flush.zero_()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        gb.attn_fwd_host(Qh_p, Kh_p, Vh_p, causal=pc.causal, window=pc.window, scale=scale_p, O=O_h, LSE=L_h,
                         device_buf=buf_p)
        e1.record(stream)
        gb.mla_decode_host(*dec_p, scale=scale_d, O=Od_h, LSE=Ld_h, device_buf=buf_d)
        e2.record(stream)
        torch.cuda.synchronize()
        if k >= e2e_warm:
            pre_ms.append(e0.elapsed_time(e1))
            e2e_pre += e0.elapsed_time(e1) / 1e3
            e2e_dec += e1.elapsed_time(e2) / 1e3
    gb.check()
    e2e_pre = max_over_ranks(e2e_pre, world)
    e2e_dec = max_over_ranks(e2e_dec, world)
    h2d_p = sum(x.numel() * x.element_size() for x in (Qh, Kh, Vh))
    d2h_p = O.numel() * 2 + LSE.numel() * 4
    h2d_d = sum(x.numel() * x.element_size() for x in dec_h)
    d2h_d = Od.numel() * 2 + Ld.numel() * 4
    # the same bytes through plain pinned copies (no kernel): what the copies alone allow
    ceil_p = copy_ceiling(dev, [Qh_p, Kh_p, Vh_p], [O_h, L_h], flush)
    ceil_d = copy_ceiling(dev, dec_p, [Od_h, Ld_h], flush)

    extra = {}
    if not args.no_extra:
        extra["prefill_workloads"] = other_prefill_workloads(gb, dev, pc.name, peaks_now(), flush)
        extra["decode_paged"] = paged_decode_workload(gb, dev, peaks_now(), flush)
        extra["decode_paged_packed"] = paged_decode_workload(gb, dev, peaks_now(), flush, H=64, s_q=2)
        extra["prefill_sparse"] = sparse_prefill_workload(gb, dev, peaks_now(), flush)
        extra["ssd_scan"] = ssd_workload(gb, dev, peaks_now(), flush)
    torch.cuda.synchronize()
    t_wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall2, timed=(t_wall0, t_wall1))

    if rank != 0:
        return
    src_p = kernel_source_hash("attn_fwd.cu")
    src_d = kernel_source_hash("mla_decode.cu")
    roof_p = {"bound": "tensor", "achieved": tflops / world, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
              "frac": tflops / world / peaks["bf16_tflops"],
              "traffic": traffic_per_launch("attn_fwd_kernel", "attn_fwd.cu", pc.name),
              "kernel": prefill_form(pc), "peak_source": f"{peak_src} bf16 dense (burst)",
              "algorithmic_flops_per_launch": fl_p}
    roof_d = {"bound": "hbm", "achieved": gbs / world, "peak": peaks["hbm_gbs"], "unit": "GB/s",
              "frac": gbs / world / peaks["hbm_gbs"],
              "traffic": traffic_per_launch("mla_decode", "mla_decode.cu", dc.name),
              "kernel": "mla_split_kernel + mla_combine_kernel", "peak_source": f"{peak_src} HBM copy",
              "algorithmic_bytes_per_launch": by_d}
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": (t_pre + t_dec) / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(pc, dc, world),
        "roofline": roof_p,
        "decode": {"metric": "MLA-decode HBM GB/s", "value": gbs, "unit": "GB/s",
                   "ms_per_launch": dec_launch_s * 1e3, "roofline": roof_d,
                   "tflops": decode_flops(dc) * args.steps * world / t_dec / 1e12,
                   "e2e": {"value": by_d * e2e_steps * world / e2e_dec / 1e9, "unit": "GB/s",
                           "h2d_bytes_per_step": h2d_d, "d2h_bytes_per_step": d2h_d}},
        "e2e": {"value": fl_p * e2e_steps * world / e2e_pre / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d_p, "d2h_bytes_per_step": d2h_p,
                "steps": e2e_steps, "warmup": e2e_warm,
                "ms_per_step_min_median_max": [min(pre_ms), sorted(pre_ms)[len(pre_ms) // 2], max(pre_ms)]},
        "e2e_ceiling": {
            "what": "the e2e bytes of one step moved by plain pinned cudaMemcpyAsync (inputs in and results "
                    "out on two streams, no kernel), and the metric that copy time alone would allow",
            "prefill": {"copy_ms": ceil_p * 1e3, "gbs": (h2d_p + d2h_p) / ceil_p / 1e9,
                        "value": fl_p * world / ceil_p / 1e12, "unit": "TFLOP/s",
                        "e2e_frac": (fl_p * e2e_steps / e2e_pre) / (fl_p / ceil_p)},
            "decode": {"copy_ms": ceil_d * 1e3, "gbs": (h2d_d + d2h_d) / ceil_d / 1e9,
                       "value": by_d * world / ceil_d / 1e9, "unit": "GB/s",
                       "e2e_frac": (by_d * e2e_steps / e2e_dec) / (by_d / ceil_d)}},
        "gpu_launches": args.steps * (1 + n_dec_launches),
        "clocks": clocks,
        "wall_s_timed_region": wall,
        "kernel_source": {"attn_fwd": src_p, "mla_decode": src_d},
    }
    line.update(extra)
    if world == 1 and not args.no_cpu_baseline:
        pcase = {"case": pc, "inputs": (Qh, Kh, Vh)}
        line["cpu_baseline"] = cpu_baseline(pcase, None, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


def run_profile_case(args, local):
    """Launch only the selected kernel(s), warmup + steps times, for ncu captures."""
    import tiled_attention_flashattention_gb300 as gb
    from tiled_attention_flashattention_gb300 import _build
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    gb.load_library()
    if args.profile == "prefill":
        pc = wl.WORKLOADS[args.workload]
        Q, K, V = (x.to(dev) for x in wl.prefill_inputs(pc))
        O = torch.empty_like(Q)
        LSE = torch.empty(pc.B, pc.H, pc.N_q, dtype=torch.float32, device=dev)
        for _ in range(args.warmup + args.steps):
            gb.attn_fwd(Q, K, V, causal=pc.causal, window=pc.window, scale=pc.softmax_scale(), O=O, LSE=LSE)
    elif args.profile == "paged-packed":
        lens, (Qn, Qp, KV, Kp, table, L) = paged_inputs(dev, H=64, s_q=2)
        ws = torch.empty(gb.mla_decode_paged_workspace_bytes(len(lens), 2, 64), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup + args.steps):
            gb.mla_decode_paged(Qn, Qp, KV, Kp, table, L, workspace=ws)
    elif args.profile == "ssd":
        c = wl.SsdCase(**{**wl.SSD_WORKLOAD.__dict__, "Bsz": args.ssd_batch or wl.SSD_WORKLOAD.Bsz})
        x, dt, A, B, C, D = (t.to(dev) for t in wl.ssd_inputs(c))
        y = torch.empty(c.Bsz, c.L, c.H, c.P, dtype=torch.float32, device=dev)
        S = torch.empty(c.Bsz, c.H, c.P, c.N, dtype=torch.float32, device=dev)
        for _ in range(args.warmup + args.steps):
            gb.ssd_scan(x, dt, A, B, C, D, y=y, final_state=S)
    else:
        dc = wl.WORKLOADS[args.decode_workload]
        Qn, Qp, KV, Kp = (x.to(dev) for x in wl.mla_inputs(dc))
        O = torch.empty(dc.B, dc.H, dc.d_c, dtype=torch.bfloat16, device=dev)
        LSE = torch.empty(dc.B, dc.H, dtype=torch.float32, device=dev)
        ws = torch.empty(max(16, gb.mla_decode_workspace_bytes(dc.B, dc.H, dc.N_kv, dc.d_c)),
                         dtype=torch.uint8, device=dev)
        for _ in range(args.warmup + args.steps):
            gb.mla_decode(Qn, Qp, KV, Kp, scale=dc.softmax_scale(), O=O, LSE=LSE, workspace=ws)
    gb.check()
    print(f"profile case {args.profile}: {args.warmup + args.steps} launches ok", flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=PREFILL, choices=[k for k, v in wl.WORKLOADS.items()
                                                            if isinstance(v, wl.PrefillCase)])
    ap.add_argument("--decode-workload", default=DECODE, choices=[k for k, v in wl.WORKLOADS.items()
                                                                  if isinstance(v, wl.MlaCase)])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other prefill workloads")
    ap.add_argument("--profile", choices=["prefill", "decode", "paged-packed", "ssd"], default=None,
                    help="only launch the selected kernel warmup+steps times (for ncu captures)")
    ap.add_argument("--ssd-batch", type=int, default=0,
                    help="with --profile ssd: batch entries of the SSD workload (default: all)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup(args.gpus)
    if args.profile:
        run_profile_case(args, local)
        return
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
