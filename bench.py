#!/usr/bin/env python
"""Benchmark of the fused online-softmax attention hot path on GB300.

One step = one pass of the whole path on synthetic bf16 inputs already
resident in HBM:
  * prefill (Rolling Update form): causal MHA, B=4, H=32, L=4096, d=128;
  * split-K decode + log-sum-exp combine (Split-K Update form): GQA,
    batch 64, 32 query / 8 KV heads, d=128, kv_len uniform in [1024, 32768].
The headline value is the prefill's attention TFLOP/s (4*d FLOPs per unmasked
query-key pair); the decode's KV GB/s (K and V bytes read once per KV head)
is reported beside it, each with its roofline against the measured GB300
peaks. All inputs are larger than L2 (129 MB), so no L2 flush is needed.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas, weak scaling); rank 0 prints one JSON line.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (prefill), KV GB/s (decode), % of GB300 roofline"
PREFILL_WORKLOAD = "prefill_mha_causal_4k"
DECODE_WORKLOAD = "decode_gqa_varlen"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------- work accounting
def causal_pairs(Lq: int, Lk: int) -> int:
    """Unmasked (query, key) pairs of one head under the bottom-right aligned
    causal mask: row i sees min(Lk, max(0, i + Lk - Lq + 1)) keys."""
    total = 0
    off = Lk - Lq
    # rows with 0 < i + off + 1 < Lk see i + off + 1 keys; later rows see Lk
    i_lo = max(0, -off)                 # first row that sees a key
    i_full = max(0, Lk - off - 1)       # first row that sees all Lk keys
    a, b = i_lo, min(Lq, i_full)
    if b > a:
        n = b - a
        first = a + off + 1
        total += n * first + n * (n - 1) // 2
    if Lq > max(i_full, i_lo):
        total += (Lq - max(i_full, i_lo)) * Lk
    return total


def prefill_flops(B, Hq, Lq, Lk, d, causal) -> int:
    """QK^T and PV: 2*d multiply-adds each per unmasked pair = 4*d FLOPs."""
    pairs = causal_pairs(Lq, Lk) if causal else Lq * Lk
    return 4 * d * B * Hq * pairs


def prefill_io_bytes(B, Hq, Hkv, Lq, Lk, d, elem=2) -> int:
    """Q read, O written, K and V read once per KV head (fused kernel)."""
    return 2 * B * Hq * Lq * d * elem + 2 * B * Hkv * Lk * d * elem


def score_round_trip_bytes(N, elem=2) -> int:
    """Unfused: the N x N score matrix written once and read once."""
    return 2 * N * N * elem


def decode_kv_bytes(Hkv, kv_lens, d, elem=2) -> int:
    """K and V of every sequence read once per KV head."""
    return sum(2 * Hkv * int(L) * d * elem for L in kv_lens)


def decode_kv_bytes_per_query_head(Hq, kv_lens, d, elem=2) -> int:
    """Ungrouped decode: every query head reads its K and V."""
    return sum(2 * Hq * int(L) * d * elem for L in kv_lens)


# -------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(relpath: str) -> str:
    with open(os.path.join(ROOT, relpath), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def recorded_traffic(kernel: str, relpath: str):
    """DRAM bytes per launch from profiles/traffic.txt, if they were taken on
    the kernel source as it is now (same digest); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    dig = source_digest(relpath)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and parts[1] == dig:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over the process group (identity when world=1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle
def oracle_prefill_sample(budget_s: float, seed: int = 0):
    """Times the fp64 oracle on the prefill workload: whole heads (each a
    seeded head of the same shape and distribution), rows taken in chunks of
    512 from the longest down, until the time budget is spent.
    Returns (flops, seconds, description)."""
    import workloads as W
    from oracle import attention_ref
    cfg = W.PREFILL_CONFIGS[PREFILL_WORKLOAD]
    rows_per_chunk = 512
    flops = 0
    nrows = 0
    heads = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        g = W.seeded_generator(cfg.seed * 1000 + seed * 100 + heads, "cpu")
        q = W._normal_bf16((1, 1, cfg.Lq, cfg.d), g, "cpu")
        k = W._normal_bf16((1, 1, cfg.Lk, cfg.d), g, "cpu")
        v = W._normal_bf16((1, 1, cfg.Lk, cfg.d), g, "cpu")
        heads += 1
        done = 0
        while done < cfg.Lq and time.perf_counter() - t0 < budget_s:
            hi = cfg.Lq - done
            lo = max(0, hi - rows_per_chunk)
            rows = list(range(lo, hi))
            attention_ref(q, k, v, scale=cfg.scale, causal=True, rows=rows)
            flops += 4 * cfg.d * sum(i + 1 for i in rows)
            done += hi - lo
        nrows += done
    dt = time.perf_counter() - t0
    desc = (f"{nrows} causal query rows over {heads} head(s) shaped like {PREFILL_WORKLOAD} "
            f"(L=4096, d=128), fp64 numpy oracle, {flops / 1e9:.1f} GFLOP")
    return flops, dt, desc


def cpu_cores() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# ---------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # each step a bounded sample; the whole run stays within a few minutes
    per_step_budget = max(0.5, min(4.0, 150.0 / (args.steps + args.warmup)))
    times, flops_all = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        fl, dt, desc = oracle_prefill_sample(per_step_budget, seed=0)
        if i >= args.warmup:
            times.append(dt)
            flops_all.append(fl)
    total_t = sum(times)
    value = sum(flops_all) / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL_WORKLOAD, "B": 4, "H": 32, "L": 4096, "d": 128,
                   "causal": True, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import online_softmax_fusion_gb300 as attn
    import workloads as W
    attn.lib()
    peaks, peak_src = load_peaks()

    pc = W.PREFILL_CONFIGS[PREFILL_WORKLOAD]
    dc = W.DECODE_CONFIGS[DECODE_WORKLOAD]
    pin = W.make_prefill_inputs(pc, dev)
    din = W.make_decode_inputs(dc, dev)
    q, k, v = pin["q"], pin["k"], pin["v"]
    O = torch.empty_like(q)
    LSE = torch.empty((pc.B, pc.Hq, pc.Lq), dtype=torch.float32, device=dev)
    S = attn.resolve_splits(dc.B, dc.Hkv, dc.Lk_max, dc.d, dc.num_splits)
    Op = torch.empty((dc.B, dc.Hq, S, dc.d), dtype=torch.float32, device=dev)
    Lp = torch.empty((dc.B, dc.Hq, S), dtype=torch.float32, device=dev)
    Od = torch.empty((dc.B, dc.Hq, dc.d), dtype=torch.bfloat16, device=dev)
    Ld = torch.empty((dc.B, dc.Hq), dtype=torch.float32, device=dev)
    kv_lens = din["kv_lens"]

    def prefill():
        attn.prefill(q, k, v, causal=True, scale=pc.scale, out=O, lse=LSE)

    def decode_part():
        attn.decode_splitk(din["q"], din["k"], din["v"], kv_lens, scale=dc.scale, num_splits=S,
                           o_part=Op, lse_part=Lp)

    def combine_part():
        attn.combine(Op, Lp, out=Od, lse=Ld)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        prefill()
        decode_part()
        combine_part()
    torch.cuda.synchronize()
    assert attn.device_status() == 0, "device status after warm-up"

    clocks = ClockSampler(dev.index).start()
    time.sleep(0.3)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        prefill()
        ev[i][1].record(stream)
        decode_part()
        ev[i][2].record(stream)
        combine_part()
        ev[i][3].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    st = attn.device_status()
    assert st == 0, f"device status {st}"

    total_ms = start.elapsed_time(end)
    t_prefill = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps   # ms per launch
    t_decode = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    t_combine = sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps
    total_ms = max_over_ranks(total_ms, world, dev)
    t_prefill_max = max_over_ranks(t_prefill, world, dev)

    fl = prefill_flops(pc.B, pc.Hq, pc.Lq, pc.Lk, pc.d, True)
    value = fl * world / (t_prefill_max * 1e-3) / 1e12            # whole job, TFLOP/s
    achieved = fl / (t_prefill * 1e-3) / 1e12
    lens = kv_lens.cpu().tolist()
    kvb = decode_kv_bytes(dc.Hkv, lens, dc.d)
    dec_gbs = kvb / (t_decode * 1e-3) / 1e9
    dec_path_gbs = kvb / ((t_decode + t_combine) * 1e-3) / 1e9

    # ----- e2e: host buffers through the public API, copies inside the region
    hq = q.cpu().pin_memory()
    hk = k.cpu().pin_memory()
    hv = v.cpu().pin_memory()
    ho = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    hl = torch.empty(LSE.shape, dtype=LSE.dtype).pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    e2e_steps = max(3, min(args.steps, 10))

    def e2e_step():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        attn.prefill(dq, dk, dv, causal=True, scale=pc.scale, out=O, lse=LSE)
        ho.copy_(O, non_blocking=True)
        hl.copy_(LSE, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e_val = fl * world / (e2e_ms * 1e-3) / 1e12
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2
    d2h = ho.numel() * 2 + hl.numel() * 4
    del hq, hk, hv, ho, hl, dq, dk, dv

    out = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cfl, cdt, cdesc = oracle_prefill_sample(args.cpu_budget)
            cpu = {"value": cfl / cdt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
                   "kind": "oracle", "sample": cdesc, "seconds": round(cdt, 2)}
        pk_t = peaks["bf16_tflops"]
        traffic = recorded_traffic("prefill", "online_softmax_fusion_gb300/csrc/prefill_tc.cu")
        dec_traffic = recorded_traffic("decode", "online_softmax_fusion_gb300/csrc/decode.cu")
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{PREFILL_WORKLOAD} + {DECODE_WORKLOAD}",
                       "prefill": {"B": pc.B, "H": pc.Hq, "L": pc.Lq, "d": pc.d, "causal": True,
                                   "flops_per_step": fl},
                       "decode": {"B": dc.B, "Hq": dc.Hq, "Hkv": dc.Hkv, "d": dc.d,
                                  "kv_len": [dc.len_lo, dc.len_hi], "splits": S,
                                  "kv_bytes_per_step": kvb},
                       "l2": "inputs larger than L2 (no flush)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk_t, "unit": "TFLOP/s",
                         "frac": achieved / pk_t, "traffic": traffic,
                         "peak_kind": f"{peak_src} bf16 burst",
                         "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "kernel": "prefill", "ms_per_launch": t_prefill},
            "decode": {"metric": "KV GB/s (decode)", "value": dec_gbs * world, "unit": "GB/s",
                       "path_value": dec_path_gbs * world,
                       "ms_decode": t_decode, "ms_combine": t_combine,
                       "roofline": {"bound": "hbm", "achieved": dec_gbs,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": dec_gbs / peaks["hbm_gbs"], "traffic": dec_traffic,
                                    "peak_kind": f"{peak_src} copy bandwidth"}},
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 3 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
