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


def window_pairs(Lq: int, Lk: int, left: int, right: int, causal: bool) -> int:
    """Unmasked (query, key) pairs of one head under a sliding window: aligned
    row i' = i + Lk - Lq sees keys [i' - left, i' + right] (a negative bound
    is unlimited on that side), and with causal keys after i' stay masked."""
    import numpy as np
    i = np.arange(Lq, dtype=np.int64) + (Lk - Lq)
    lo = np.zeros_like(i) if left < 0 else np.maximum(0, i - left)
    hi = np.full_like(i, Lk - 1)
    if right >= 0:
        hi = np.minimum(hi, i + right)
    if causal:
        hi = np.minimum(hi, i)
    return int(np.maximum(0, hi - lo + 1).sum())


def backward_flops(B, Hq, Lq, Lk, d, causal) -> int:
    """Five products per unmasked pair (S recomputed, dP, dV, dK, dQ): 10*d."""
    pairs = causal_pairs(Lq, Lk) if causal else Lq * Lk
    return 10 * d * B * Hq * pairs


def rmsnorm_matmul_bytes(B, H, D) -> int:
    """Algorithmic bytes of O = RMSNorm(X; G) W: W, X and G read once, O written once (bf16)."""
    return 2 * (H * D + B * H + H + B * D)


def rmsnorm_matmul_flops(B, H, D) -> int:
    return 2 * B * H * D


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
    """nvidia-smi clock / throttle sampling in the background; stop() keeps
    the samples whose timestamps fall inside the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

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
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    @staticmethod
    def _epoch(ts: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(ts.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    @classmethod
    def summarize(cls, lines, t0=None, t1=None):
        rows = []
        for line in lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 10:
                continue
            ts = cls._epoch(p[0])
            rows.append((ts, p))
        inside = [p for ts, p in rows
                  if t0 is None or (ts is not None and t0 - 0.025 <= ts <= t1 + 0.025)]
        use = inside if inside else [p for _, p in rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[2]) for r in use) if v is not None]
        mx = [v for v in (num(r[3]) for r in use) if v is not None]
        pw = [v for v in (num(r[4]) for r in use) if v is not None]
        reasons = sorted({cls.REASONS[i] for r in use for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples_in_region": len(inside), "samples": len(rows),
                "power_w_max": max(pw) if pw else None}

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return self.summarize(lines, t0, t1)


class NvmlSampler:
    """Samples the SM clock, the clock-event (throttle) reasons and the power
    of one GPU through NVML (read-only queries, ctypes) every `period_s` in a
    background thread, so that a timed region of a few milliseconds still
    holds tens of samples. stop(t0, t1) keeps the samples taken inside
    [t0, t1] (time.time() seconds)."""
    SM_CLOCK = 1
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, uuid: str | None = None, period_s: float = 0.0005):
        import ctypes
        self.ct = ctypes
        self.period = period_s
        self.samples = []
        self.thread = None
        self.stop_flag = False
        self.ok = False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            found = False
            if uuid:
                found = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            if not found:
                found = lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0
            if not found:
                return
            self.lib, self.h = lib, h
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, self.SM_CLOCK, ctypes.byref(mx))
            self.max_mhz = float(mx.value)
            self.ok = True
        except Exception:
            self.ok = False

    def _sample(self):
        ct = self.ct
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        t = time.time()
        self.lib.nvmlDeviceGetClockInfo(self.h, self.SM_CLOCK, ct.byref(clk))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
        self.reasons_fn(self.h, ct.byref(rs))
        self.samples.append((t, float(clk.value), pw.value / 1000.0, int(rs.value)))

    def _run(self):
        while not self.stop_flag:
            self._sample()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            import threading
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    @classmethod
    def summarize(cls, samples, max_mhz, t0=None, t1=None):
        inside = [s for s in samples if t0 is None or t0 <= s[0] <= t1]
        sm = [s[1] for s in inside]
        reasons = sorted({name for s in inside for bit, name in cls.REASON_BITS.items()
                          if s[3] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max_mhz,
                "reasons": reasons, "samples_in_region": len(inside), "samples": len(samples),
                "power_w_max": max((s[2] for s in inside), default=None),
                "sm_mhz_min": min(sm) if sm else None, "source": "nvml"}

    def stop(self, t0=None, t1=None):
        self.stop_flag = True
        if self.thread is not None:
            self.thread.join(timeout=2)
        return self.summarize(self.samples, self.max_mhz, t0, t1)


def start_clock_sampler(dev):
    """NVML sampling when the library is there, nvidia-smi otherwise."""
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    s = NvmlSampler(dev.index, uuid)
    if s.ok:
        return s.start()
    return ClockSampler(dev.index).start()


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


def time_launches(fn, steps, warmup, stream):
    """Mean CUDA-event time (ms) of fn() over `steps` launches after warm-up."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def graph_time(fn, reps, replays=5):
    """Mean time (ms) of fn() replayed from a CUDA graph of `reps` calls, so
    short kernels are timed without the host's per-call overhead. The first
    call runs outside capture (it sets kernel attributes and looks up the
    status word's address)."""
    import torch
    fn()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                fn()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(replays):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (replays * reps)


def prefill_check_sample(name, q, k, v, O, LSE, heads, rows, G, scale, causal=True,
                         slopes=None, softcap=0.0, window=(-1, -1)):
    """Host copies of what the oracle needs to check some rows of some heads
    of a prefill output: the heads' query rows, their K/V heads and the
    kernel's O / LSE rows."""
    import torch
    idx = torch.as_tensor(rows, dtype=torch.int64, device=q.device)
    items = []
    for b, h in heads:
        kv = h // G
        items.append({"q": q[b, h].index_select(0, idx).cpu(), "k": k[b, kv].cpu(),
                      "v": v[b, kv].cpu(), "O": O[b, h].index_select(0, idx).cpu(),
                      "LSE": LSE[b, h].index_select(0, idx).cpu(),
                      "slope": None if slopes is None else float(slopes[h])})
    return {"workload": name, "kind": "prefill", "rows": list(rows), "Lq": int(q.shape[2]),
            "items": items, "scale": scale, "causal": causal, "softcap": softcap,
            "window": window}


def decode_check_sample(name, q, k, v, lens, O, LSE, pairs, G, scale):
    """Host copies for an oracle check of some (batch entry, KV head) groups
    of a decode output."""
    items = []
    for b, kvh in pairs:
        n = int(lens[b])
        items.append({"q": q[b, kvh * G:(kvh + 1) * G].cpu(), "k": k[b, kvh, :n].cpu(),
                      "v": v[b, kvh, :n].cpu(), "O": O[b, kvh * G:(kvh + 1) * G].cpu(),
                      "LSE": LSE[b, kvh * G:(kvh + 1) * G].cpu()})
    return {"workload": name, "kind": "decode", "items": items, "scale": scale}


def measure_other_workloads(attn, W, dev, peaks, checks):
    """The remaining workloads, each timed on its own (inputs > L2 except the
    smallest sweep lengths, which are noted): the causal GQA + ALiBi prefill
    sweep over L and the long-context outlier decode with 64 splits. A small
    sample of each output is appended to `checks` for the oracle leg."""
    import torch
    stream = torch.cuda.current_stream()
    sweep = []
    for L in W.GQA_SWEEP_LENGTHS:
        cfg = W.gqa_sweep_config(L)
        inp = W.make_prefill_inputs(cfg, dev)
        O = torch.empty_like(inp["q"])
        LSE = torch.empty((cfg.B, cfg.Hq, cfg.Lq), dtype=torch.float32, device=dev)
        fn = lambda: attn.prefill(inp["q"], inp["k"], inp["v"], causal=True, scale=cfg.scale,  # noqa: E731
                                  alibi_slopes=inp["alibi_slopes"], out=O, lse=LSE)
        # replayed from a CUDA graph: the short lengths would otherwise time
        # the host's per-call overhead rather than the kernel
        ms = graph_time(fn, 10 if L <= 8192 else 2, replays=5 if L <= 16384 else 2)
        fl = prefill_flops(cfg.B, cfg.Hq, cfg.Lq, cfg.Lk, cfg.d, True)
        tf = fl / (ms * 1e-3) / 1e12
        in_bytes = (inp["q"].numel() + inp["k"].numel() + inp["v"].numel()) * 2
        sweep.append({"L": L, "ms": ms, "tflops": tf, "frac": tf / peaks["bf16_tflops"],
                      "inputs_exceed_l2": in_bytes > 129e6, "timing": "cuda graph replay"})
        rows = W.sample_rows(L, 24, 4, L).tolist()
        checks.append(prefill_check_sample(cfg.name, inp["q"], inp["k"], inp["v"], O, LSE,
                                           [(0, 0), (0, 31)], rows, cfg.Hq // cfg.Hkv,
                                           cfg.scale, slopes=inp["alibi_slopes"].cpu()))
        del inp, O, LSE
    # SoftCap and a causal sliding window on the causal MHA workload
    pc = W.PREFILL_CONFIGS[PREFILL_WORKLOAD]
    pin = W.make_prefill_inputs(pc, dev)
    Ov = torch.empty_like(pin["q"])
    Lv = torch.empty((pc.B, pc.Hq, pc.Lq), dtype=torch.float32, device=dev)
    variants = []
    for name, cap, win in (("softcap_30", 30.0, (-1, -1)), ("window_left_1024", 0.0, (1024, -1))):
        ms = graph_time(lambda: attn.prefill(pin["q"], pin["k"], pin["v"], causal=True,
                                             scale=pc.scale, out=Ov, lse=Lv, softcap=cap,
                                             window=win), 4, replays=3)
        pairs = window_pairs(pc.Lq, pc.Lk, win[0], win[1], True)
        fl = 4 * pc.d * pc.B * pc.Hq * pairs
        tf = fl / (ms * 1e-3) / 1e12
        variants.append({"variant": name, "ms": ms, "tflops": tf,
                         "frac": tf / peaks["bf16_tflops"], "flops": fl,
                         "workload": PREFILL_WORKLOAD, "timing": "cuda graph replay"})
        rows = W.sample_rows(pc.Lq, 24, 4, 7).tolist()
        checks.append(prefill_check_sample(f"{PREFILL_WORKLOAD} {name}", pin["q"], pin["k"],
                                           pin["v"], Ov, Lv, [(1, 5)], rows, 1, pc.scale,
                                           softcap=cap, window=win))
    del pin, Ov, Lv
    # backward of the causal MHA workload (forward outputs as its inputs)
    pc = W.PREFILL_CONFIGS[PREFILL_WORKLOAD]
    pin = W.make_prefill_inputs(pc, dev)
    g = W.seeded_generator(pc.seed + 7, dev)
    dout = W._normal_bf16(pin["q"].shape, g, dev)
    O, LSE = attn.prefill(pin["q"], pin["k"], pin["v"], causal=True, scale=pc.scale)
    ws = torch.empty(attn.lib().attn_backward_workspace_bytes(pc.B, pc.Hq, pc.Lq, pc.d) // 4,
                     dtype=torch.float32, device=dev)
    t_bwd = time_launches(lambda: attn.backward(pin["q"], pin["k"], pin["v"], O, LSE, dout,
                                                causal=True, scale=pc.scale, workspace=ws),
                          5, 2, stream)
    bfl = backward_flops(pc.B, pc.Hq, pc.Lq, pc.Lk, pc.d, True)
    bwd = {"workload": PREFILL_WORKLOAD + " backward", "ms": t_bwd,
           "tflops": bfl / (t_bwd * 1e-3) / 1e12,
           "frac": bfl / (t_bwd * 1e-3) / 1e12 / peaks["bf16_tflops"],
           "flops": bfl, "kernels": "prep + main (tcgen05) + convert"}
    del pin, dout, O, LSE, ws
    dc = W.DECODE_CONFIGS["decode_long_outlier"]
    din = W.make_decode_inputs(dc, dev)
    S = attn.resolve_splits(dc.B, dc.Hkv, dc.Lk_max, dc.d, dc.num_splits)
    Op = torch.empty((dc.B, dc.Hq, S, dc.d), dtype=torch.float32, device=dev)
    Lp = torch.empty((dc.B, dc.Hq, S), dtype=torch.float32, device=dev)
    Od = torch.empty((dc.B, dc.Hq, dc.d), dtype=torch.bfloat16, device=dev)
    Ld = torch.empty((dc.B, dc.Hq), dtype=torch.float32, device=dev)
    t_dec = time_launches(lambda: attn.decode_splitk(din["q"], din["k"], din["v"], din["kv_lens"],
                                                     scale=dc.scale, num_splits=S, o_part=Op,
                                                     lse_part=Lp), 10, 3, stream)
    t_cmb = time_launches(lambda: attn.combine(Op, Lp, out=Od, lse=Ld), 10, 3, stream)
    kvb = decode_kv_bytes(dc.Hkv, din["kv_lens"].cpu().tolist(), dc.d)
    gbs = kvb / (t_dec * 1e-3) / 1e9
    long_dec = {"workload": dc.name, "splits": S, "ms_decode": t_dec, "ms_combine": t_cmb,
                "kv_gbs": gbs, "path_gbs": kvb / ((t_dec + t_cmb) * 1e-3) / 1e9,
                "frac": gbs / peaks["hbm_gbs"], "kv_bytes": kvb}
    checks.append(decode_check_sample(dc.name, din["q"], din["k"], din["v"],
                                      din["kv_lens"].cpu().tolist(), Od, Ld, [(0, 0), (3, 7)],
                                      dc.Hq // dc.Hkv, dc.scale))
    del din, Op, Lp, Od, Ld
    # fused RMSNorm + product at the LLaMA-2-7B shape (H = D = 4096): the calls
    # cycle through 5 copies of W (5 x 32 MB > L2), so each reads W from HBM
    rms = []
    for name in ("rmsnorm_matmul_llama7b_b16", "rmsnorm_matmul_llama7b_b256"):
        cfg = W.RMS_MATMUL_CONFIGS[name]
        rin = W.make_rmsnorm_matmul_inputs(cfg, dev)
        wcopies = [rin["w"]] + [rin["w"].clone() for _ in range(4)]
        Orm = torch.empty((cfg.B, cfg.D), dtype=torch.bfloat16, device=dev)

        wsb = torch.empty((attn.rmsnorm_matmul_ws_bytes(cfg.B, cfg.H),), dtype=torch.uint8,
                          device=dev)

        def fn_rms(chained):
            for wc in wcopies:
                attn.rmsnorm_matmul(rin["x"], rin["g"], wc, out=Orm, chained=chained)

        def fn_ws(chained=False):
            for wc in wcopies:
                attn.rmsnorm_matmul(rin["x"], rin["g"], wc, out=Orm, form="auto", workspace=wsb,
                                    chained=chained)
        ms_plain = graph_time(lambda: fn_rms(False), 4, replays=5) / len(wcopies)
        # a stack of calls with constant weights: each launch overlaps the
        # end of the one before (programmatic dependent launch)
        ms_chained = graph_time(lambda: fn_rms(True), 4, replays=5) / len(wcopies)
        # the workspace entry (two-pass form), plainly and chained
        ms_ws = graph_time(fn_ws, 4, replays=5) / len(wcopies)
        ms_ws_chained = graph_time(lambda: fn_ws(True), 4, replays=5) / len(wcopies)
        forms = {"chained": ms_chained, "two_pass": ms_ws, "two_pass_chained": ms_ws_chained}
        form = min(forms, key=forms.get)
        ms = forms[form]
        byts = rmsnorm_matmul_bytes(cfg.B, cfg.H, cfg.D)
        fl = rmsnorm_matmul_flops(cfg.B, cfg.H, cfg.D)
        gbs = byts / (ms * 1e-3) / 1e9
        tf = fl / (ms * 1e-3) / 1e12
        rms.append({"workload": name, "B": cfg.B, "H": cfg.H, "D": cfg.D, "ms": ms,
                    "gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "tflops": tf,
                    "frac_bf16": tf / peaks["bf16_tflops"], "bytes": byts, "flops": fl,
                    "splits": attn.lib().attn_rmsnorm_matmul_splits(cfg.B, cfg.H, cfg.D),
                    "ms_single_launch": ms_plain, "ms_chained": ms_chained,
                    "ms_workspace_entry": ms_ws, "ms_workspace_entry_chained": ms_ws_chained,
                    "form": form,
                    "timing": "cuda graph replay of 5 back-to-back calls, W rotated over 5 "
                              "copies (> L2); ms = the fastest of the chained fused calls and "
                              "the workspace entry, plain or chained (form names it); "
                              "ms_single_launch: plain fused calls"})
        checks.append({"workload": name, "kind": "rmsnorm", "x": rin["x"][:3].cpu(),
                       "g": rin["g"].cpu(), "w": rin["w"].cpu(), "O": Orm[:3].cpu()})
        del rin, wcopies, Orm
    return {"prefill_gqa_alibi_sweep": sweep, "decode_long_outlier": long_dec,
            "backward_causal_mha_4k": bwd, "rmsnorm_matmul": rms,
            "prefill_softcap_window": variants}


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


class ErrorStats:
    """Max / mean absolute error of outputs against the oracle, per workload."""

    def __init__(self):
        self.acc = {}

    def add(self, name, O, Or, L=None, Lr=None):
        import numpy as np
        o = np.asarray(O.float().numpy() if hasattr(O, "float") else O, dtype=np.float64)
        e = np.abs(o - np.asarray(Or, dtype=np.float64))
        a = self.acc.setdefault(name, {"o_max_abs": 0.0, "o_sum": 0.0, "o_n": 0,
                                       "lse_max_abs": 0.0, "rows": 0, "empty_rows_exact": True})
        a["o_max_abs"] = max(a["o_max_abs"], float(e.max(initial=0.0)))
        a["o_sum"] += float(e.sum())
        a["o_n"] += e.size
        if L is not None:
            lg = np.asarray(L.numpy() if hasattr(L, "numpy") else L, dtype=np.float64)
            lr = np.asarray(Lr, dtype=np.float64)
            fin = np.isfinite(lr)
            if fin.any():
                a["lse_max_abs"] = max(a["lse_max_abs"], float(np.abs(lg[fin] - lr[fin]).max()))
            empty = np.isneginf(lr)
            if empty.any():
                a["empty_rows_exact"] &= bool(np.all(np.isneginf(lg[empty])) and
                                              np.all(o[empty] == 0.0))
            a["rows"] += lr.size

    def summary(self):
        out = {}
        for name, a in self.acc.items():
            out[name] = {"o_max_abs": a["o_max_abs"],
                         "o_mean_abs": a["o_sum"] / max(1, a["o_n"]),
                         "lse_max_abs": a["lse_max_abs"], "rows": a["rows"],
                         "empty_rows_exact": a["empty_rows_exact"]}
        return out


def oracle_leg(budget_s, prefill_ctx, decode_ctx, checks, dec_budget_s):
    """The CPU oracle beside the kernels, on the bench's own inputs: times it
    on the prefill workload (whole heads, rows in chunks of 512 from the
    longest down, until budget_s is spent) and on the decode workload ((batch
    entry, KV head) groups in order until dec_budget_s), and compares every
    row it computes with the kernels' output of the timed steps; then checks
    the samples the other workloads left in `checks`, and the single-head
    workload. Returns (cpu_baseline dict, per-workload error stats)."""
    import torch
    import online_softmax_fusion_gb300 as attn
    import workloads as W
    from oracle import attention_ref, decode_ref, rmsnorm_matmul_ref
    errs = ErrorStats()
    cpu = {"kind": "oracle", "cores": cpu_cores(), "unit": "TFLOP/s"}
    if prefill_ctx is not None:
        pc = prefill_ctx["cfg"]
        q, k, v, O, LSE = (prefill_ctx[x] for x in ("q", "k", "v", "O", "LSE"))
        heads = [(b, h) for h in range(pc.Hq) for b in range(pc.B)]
        flops = nrows = 0
        t_or = 0.0
        for (b, h) in heads:
            if t_or >= budget_s:
                break
            qh, kh, vh = q[b:b + 1, h:h + 1].cpu(), k[b:b + 1, h:h + 1].cpu(), v[b:b + 1, h:h + 1].cpu()
            Oh, Lh = O[b, h].cpu(), LSE[b, h].cpu()
            done = 0
            while done < pc.Lq and t_or < budget_s:
                hi = pc.Lq - done
                lo = max(0, hi - 512)
                rows = list(range(lo, hi))
                t0 = time.perf_counter()
                Or, Lr = attention_ref(qh, kh, vh, scale=pc.scale, causal=True, rows=rows)
                t_or += time.perf_counter() - t0
                errs.add(pc.name, Oh[lo:hi], Or[0, 0], Lh[lo:hi], Lr[0, 0])
                flops += 4 * pc.d * sum(i + 1 for i in rows)
                nrows += hi - lo
                done += hi - lo
        cpu.update({"value": flops / t_or / 1e12, "seconds": round(t_or, 2),
                    "sample": f"{nrows} causal rows of {pc.name} (its own inputs), "
                              f"{flops / 1e9:.0f} GFLOP, fp64 numpy"})
    if decode_ctx is not None:
        dc = decode_ctx["cfg"]
        q, k, v, lens, O, LSE = (decode_ctx[x] for x in ("q", "k", "v", "lens", "O", "LSE"))
        G = dc.Hq // dc.Hkv
        kvb = 0
        t_or = 0.0
        groups = 0
        for b in range(dc.B):
            for kvh in range(dc.Hkv):
                if t_or >= dec_budget_s:
                    break
                n = int(lens[b])
                qg = q[b:b + 1, kvh * G:(kvh + 1) * G].cpu()
                kg, vg = k[b:b + 1, kvh:kvh + 1, :n].cpu(), v[b:b + 1, kvh:kvh + 1, :n].cpu()
                t0 = time.perf_counter()
                Or, Lr = decode_ref(qg, kg, vg, [n], scale=dc.scale)
                t_or += time.perf_counter() - t0
                errs.add(dc.name, O[b, kvh * G:(kvh + 1) * G].cpu(), Or[0],
                         LSE[b, kvh * G:(kvh + 1) * G].cpu(), Lr[0])
                kvb += 2 * n * dc.d * 2
                groups += 1
        cpu.update({"decode_value": kvb / t_or / 1e9, "decode_unit": "GB/s",
                    "decode_seconds": round(t_or, 2),
                    "decode_sample": f"{groups} (batch, KV head) groups of {dc.name} (its own "
                                     f"inputs), {kvb / 1e9:.2f} GB of K/V, fp64 numpy"})
    # the single-head workload: tiny, run here in full
    c1 = W.PREFILL_CONFIGS["single_head_noncausal"]
    inp = W.make_prefill_inputs(c1, "cpu")
    O1, L1 = attn.prefill(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), causal=False,
                          scale=c1.scale)
    Or, Lr = attention_ref(inp["q"], inp["k"], inp["v"], scale=c1.scale)
    errs.add(c1.name, O1.cpu(), Or, L1.cpu(), Lr)
    for c in checks:
        if c["kind"] == "prefill":
            for it in c["items"]:
                rows = c["rows"]
                qfull = torch.zeros((1, 1, c["Lq"], it["q"].shape[-1]), dtype=it["q"].dtype)
                qfull[0, 0, rows] = it["q"]
                Or, Lr = attention_ref(qfull, it["k"][None, None], it["v"][None, None],
                                       scale=c["scale"], causal=c["causal"],
                                       alibi_slopes=None if it["slope"] is None
                                       else torch.tensor([it["slope"]]),
                                       rows=rows, softcap=c["softcap"],
                                       window_left=c["window"][0], window_right=c["window"][1])
                errs.add(c["workload"], it["O"], Or[0, 0], it["LSE"], Lr[0, 0])
        elif c["kind"] == "decode":
            for it in c["items"]:
                n = it["k"].shape[0]
                Or, Lr = decode_ref(it["q"][None], it["k"][None, None], it["v"][None, None], [n],
                                    scale=c["scale"])
                errs.add(c["workload"], it["O"], Or[0], it["LSE"], Lr[0])
        elif c["kind"] == "rmsnorm":
            ref = rmsnorm_matmul_ref(c["x"], c["g"], c["w"])
            errs.add(c["workload"], c["O"], ref)
    summ = errs.summary()
    if summ:
        cpu["err_o_max_abs"] = max(v["o_max_abs"] for k, v in summ.items()
                                   if not k.startswith("rmsnorm"))
        cpu["err_o_mean_abs_worst"] = max(v["o_mean_abs"] for k, v in summ.items()
                                          if not k.startswith("rmsnorm"))
        cpu["err_lse_max_abs"] = max(v["lse_max_abs"] for v in summ.values())
        cpu["err_workloads"] = len(summ)
    return cpu, summ


def cpu_cores() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# ---------------------------------------------------------- reference arm
def bench_config(kernel, pc, dc, world):
    """The workload description both arms print (identical for the same run)."""
    workload = {"all": f"{pc.name} + {dc.name}", "prefill": pc.name, "decode": dc.name}[kernel]
    return {"workload": workload,
            "prefill": {"B": pc.B, "H": pc.Hq, "L": pc.Lq, "d": pc.d, "causal": True}
            if kernel in ("all", "prefill") else None,
            "decode": {"B": dc.B, "Hq": dc.Hq, "Hkv": dc.Hkv, "d": dc.d,
                       "kv_len": [dc.len_lo, dc.len_hi]} if kernel in ("all", "decode") else None,
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}


def run_reference(args):
    import workloads as W
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
        "config": bench_config("all", W.PREFILL_CONFIGS[PREFILL_WORKLOAD],
                               W.DECODE_CONFIGS[DECODE_WORKLOAD], world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------- RMSNorm + MatMul only
def run_rmsnorm(args):
    """Times the fused RMSNorm + product alone at the LLaMA-2-7B shape
    (H = D = 4096) with --batch rows: `warmup` untimed then `steps` timed
    launches, each reading one of 5 copies of W in turn (5 x 32 MB > L2)."""
    import torch
    import online_softmax_fusion_gb300 as attn
    import workloads as W
    attn.lib()
    peaks, _ = load_peaks()
    cfg = W.RmsMatmulConfig(f"rmsnorm_matmul_llama7b_b{args.batch}", B=args.batch, H=4096,
                            D=4096, seed=1301)
    rin = W.make_rmsnorm_matmul_inputs(cfg, "cuda")
    wcopies = [rin["w"]] + [rin["w"].clone() for _ in range(4)]
    O = torch.empty((cfg.B, cfg.D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    it = [0]

    wsb = torch.empty((attn.rmsnorm_matmul_ws_bytes(cfg.B, cfg.H),), dtype=torch.uint8,
                      device="cuda")

    def step():
        if args.rms_form:
            attn.rmsnorm_matmul(rin["x"], rin["g"], wcopies[it[0] % 5], out=O,
                                form=args.rms_form, workspace=wsb)
        else:
            attn.rmsnorm_matmul(rin["x"], rin["g"], wcopies[it[0] % 5], out=O)
        it[0] += 1
    ms = time_launches(step, args.steps, args.warmup, stream)
    byts = rmsnorm_matmul_bytes(cfg.B, cfg.H, cfg.D)
    fl = rmsnorm_matmul_flops(cfg.B, cfg.H, cfg.D)
    gbs = byts / (ms * 1e-3) / 1e9
    print(json.dumps({"metric": "RMSNorm+MatMul GB/s", "value": gbs, "unit": "GB/s",
                      "workload": cfg.name, "ms_per_launch": ms,
                      "form": args.rms_form or "fused (single kernel)",
                      "frac_hbm": gbs / peaks["hbm_gbs"],
                      "tflops": fl / (ms * 1e-3) / 1e12, "steps": args.steps,
                      "warmup": args.warmup, "timing": "eager launches, CUDA events"}),
          flush=True)
    return 0


# ------------------------------------------------------- backward only
def run_backward(args):
    """Times the attention backward alone on the causal MHA shape (H = 32,
    L = 4096, d = 128) with --batch sequences: O and LSE from one forward,
    then `warmup` untimed and `steps` timed backward calls."""
    import torch
    import online_softmax_fusion_gb300 as attn
    import workloads as W
    attn.lib()
    peaks, _ = load_peaks()
    base = W.PREFILL_CONFIGS[PREFILL_WORKLOAD]
    cfg = W.PrefillConfig(f"{base.name}_b{args.batch}", B=args.batch, Hq=base.Hq, Hkv=base.Hkv,
                          Lq=base.Lq, Lk=base.Lk, d=base.d, causal=True, seed=base.seed)
    inp = W.make_prefill_inputs(cfg, "cuda")
    q, k, v = inp["q"], inp["k"], inp["v"]
    dout = W._normal_bf16(q.shape, W.seeded_generator(cfg.seed + 7, "cuda"), "cuda")
    O, LSE = attn.prefill(q, k, v, causal=True, scale=cfg.scale)
    ws = torch.empty(attn.lib().attn_backward_workspace_bytes(cfg.B, cfg.Hq, cfg.Lq, cfg.d) // 4,
                     dtype=torch.float32, device="cuda")
    ms = time_launches(lambda: attn.backward(q, k, v, O, LSE, dout, causal=True, scale=cfg.scale,
                                             workspace=ws),
                       args.steps, args.warmup, torch.cuda.current_stream())
    fl = backward_flops(cfg.B, cfg.Hq, cfg.Lq, cfg.Lk, cfg.d, True)
    tf = fl / (ms * 1e-3) / 1e12
    print(json.dumps({"metric": "attention backward TFLOP/s", "value": tf, "unit": "TFLOP/s",
                      "workload": cfg.name, "ms_per_call": ms,
                      "frac": tf / peaks["bf16_tflops"], "steps": args.steps,
                      "warmup": args.warmup, "kernels": "prep + main + convert"}), flush=True)
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
    do_p = args.kernel in ("all", "prefill")
    do_d = args.kernel in ("all", "decode")

    pc = W.PREFILL_CONFIGS[PREFILL_WORKLOAD]
    dc = W.DECODE_CONFIGS[DECODE_WORKLOAD]
    if args.small:
        # same distributions, smaller batches for profiling captures: ~2 GB of
        # K/V for the decode, one sequence (134 MB of Q/K/V) for the prefill
        dc = W.DecodeConfig(dc.name + "_b16", B=16, Hq=dc.Hq, Hkv=dc.Hkv, Lk_max=dc.Lk_max,
                            d=dc.d, len_lo=dc.len_lo, len_hi=dc.len_hi, seed=dc.seed)
        pc = W.PrefillConfig(pc.name + "_b1", B=1, Hq=pc.Hq, Hkv=pc.Hkv, Lq=pc.Lq, Lk=pc.Lk,
                             d=pc.d, causal=pc.causal, seed=pc.seed)
    launches = []
    if do_p:
        pin = W.make_prefill_inputs(pc, dev)
        q, k, v = pin["q"], pin["k"], pin["v"]
        O = torch.empty_like(q)
        LSE = torch.empty((pc.B, pc.Hq, pc.Lq), dtype=torch.float32, device=dev)

        def prefill():
            attn.prefill(q, k, v, causal=True, scale=pc.scale, out=O, lse=LSE,
                         softcap=args.softcap)
        launches.append(("prefill", prefill))
    if do_d:
        din = W.make_decode_inputs(dc, dev)
        S = attn.resolve_splits(dc.B, dc.Hkv, dc.Lk_max, dc.d, dc.num_splits)
        Op = torch.empty((dc.B, dc.Hq, S, dc.d), dtype=torch.float32, device=dev)
        Lp = torch.empty((dc.B, dc.Hq, S), dtype=torch.float32, device=dev)
        Od = torch.empty((dc.B, dc.Hq, dc.d), dtype=torch.bfloat16, device=dev)
        Ld = torch.empty((dc.B, dc.Hq), dtype=torch.float32, device=dev)
        kv_lens = din["kv_lens"]

        def decode_part():
            attn.decode_splitk(din["q"], din["k"], din["v"], kv_lens, scale=dc.scale,
                               num_splits=S, o_part=Op, lse_part=Lp)

        def combine_part():
            attn.combine(Op, Lp, out=Od, lse=Ld)
        launches += [("decode", decode_part), ("combine", combine_part)]

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for _, fn in launches:
            fn()
    torch.cuda.synchronize()
    assert attn.device_status() == 0, "device status after warm-up"

    clocks = start_clock_sampler(dev)
    time.sleep(0.5)   # let nvidia-smi start sampling before the region opens
    nl = len(launches)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        for li, (_, fn) in enumerate(launches):
            fn()
            ev[i][li + 1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    st = attn.device_status()
    assert st == 0, f"device status {st}"

    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    per = {}
    for li, (name, _) in enumerate(launches):
        per[name] = sum(e[li].elapsed_time(e[li + 1]) for e in ev) / args.steps  # ms per launch

    fl = prefill_flops(pc.B, pc.Hq, pc.Lq, pc.Lk, pc.d, True)
    value = achieved = None
    if do_p:
        t_prefill_max = max_over_ranks(per["prefill"], world, dev)
        value = fl * world / (t_prefill_max * 1e-3) / 1e12            # whole job, TFLOP/s
        achieved = fl / (per["prefill"] * 1e-3) / 1e12
    decode_obj = None
    kvb = None
    if do_d:
        lens = kv_lens.cpu().tolist()
        kvb = decode_kv_bytes(dc.Hkv, lens, dc.d)
        dec_gbs = kvb / (per["decode"] * 1e-3) / 1e9
        dec_path_gbs = kvb / ((per["decode"] + per["combine"]) * 1e-3) / 1e9
        dec_traffic = recorded_traffic("decode", "online_softmax_fusion_gb300/csrc/decode.cu")
        decode_obj = {"metric": "KV GB/s (decode)", "value": dec_gbs * world, "unit": "GB/s",
                      "path_value": dec_path_gbs * world, "ms_decode": per["decode"],
                      "ms_combine": per["combine"], "workload": dc.name,
                      "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                                   "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                                   "traffic": dec_traffic,
                                   "peak_kind": f"{peak_src} copy bandwidth"}}
        if not do_p:
            value = dec_gbs * world

    # ----- e2e: host buffers through the public API, copies inside the region
    e2e = None
    if do_p:
        hq = q.cpu().pin_memory()
        hk = k.cpu().pin_memory()
        hv = v.cpu().pin_memory()
        ho = torch.empty(O.shape, dtype=O.dtype).pin_memory()
        hl = torch.empty(LSE.shape, dtype=LSE.dtype).pin_memory()
        ws = attn.prefill_host_workspace(pc.B, pc.Hq, pc.Hkv, pc.Lq, pc.Lk, pc.d, dev)
        e2e_steps = max(3, min(args.steps, 10))

        def e2e_step():
            # the library's host-buffer entry: chunked copies in, kernels,
            # copies out, pipelined across streams
            attn.prefill_host(hq, hk, hv, causal=True, scale=pc.scale, out=ho, lse=hl,
                              workspace=ws, synchronize=False)

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
        # the host link's own ceiling for the same bytes: the step's copies
        # alone (no kernels), inputs in on one stream while the outputs go
        # out on another, as the pipelined entry overlaps them
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def copies_only():
            with torch.cuda.stream(s_in):
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
            with torch.cuda.stream(s_out):
                ho.copy_(O, non_blocking=True)
                hl.copy_(LSE, non_blocking=True)
        copies_only()
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(e2e_steps):
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            copies_only()
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)
        c1.record(stream)
        torch.cuda.synchronize()
        link_ms = c0.elapsed_time(c1) / e2e_steps
        e2e = {"value": fl * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": (hq.numel() + hk.numel() + hv.numel()) * 2,
               "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4, "ms_per_step": e2e_ms,
               "copies_only_ms": link_ms, "of_copies_only": link_ms / e2e_ms}
        del hq, hk, hv, ho, hl, ws

    others = None
    checks = []
    if args.kernel == "all" and not args.no_other_workloads:
        others = measure_other_workloads(attn, W, dev, peaks, checks)

    if rank == 0:
        cpu = errors = None
        if world == 1 and not args.no_cpu_baseline:
            pctx = {"cfg": pc, "q": q, "k": k, "v": v, "O": O, "LSE": LSE} if do_p else None
            dctx = {"cfg": dc, "q": din["q"], "k": din["k"], "v": din["v"],
                    "lens": kv_lens.cpu().tolist(), "O": Od, "LSE": Ld} if do_d else None
            cpu, errors = oracle_leg(args.cpu_budget, pctx, dctx, checks,
                                     args.cpu_budget / 3)
        pk_t = peaks["bf16_tflops"]
        roof = None
        if do_p:
            roof = {"bound": "tensor", "achieved": achieved, "peak": pk_t, "unit": "TFLOP/s",
                    "frac": achieved / pk_t,
                    "traffic": recorded_traffic("prefill",
                                                "online_softmax_fusion_gb300/csrc/prefill_tc.cuh"),
                    "peak_kind": f"{peak_src} bf16 burst",
                    "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                    "kernel": "prefill_tc_kernel", "ms_per_launch": per["prefill"]}
            if do_d:
                # the decode's own roofline (HBM-bound), as plain keys beside it
                dr = decode_obj["roofline"]
                roof.update({"decode_kernel": "decode_splitk_kernel",
                             "decode_bound": "hbm", "decode_achieved_gbs": dr["achieved"],
                             "decode_peak_gbs": dr["peak"], "decode_frac": dr["frac"],
                             "decode_traffic": dr["traffic"],
                             "decode_kv_bytes": kvb, "decode_ms_per_launch": per["decode"],
                             "combine_ms_per_launch": per["combine"]})
        elif do_d:
            roof = decode_obj["roofline"]
        out = {
            "metric": METRIC, "value": value,
            "unit": "TFLOP/s" if do_p else "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(bench_config(args.kernel, pc, dc, world),
                           **({"softcap": args.softcap} if args.softcap else {})),
            "roofline": roof,
            "decode": decode_obj,
            "e2e": e2e,
            "gpu_launches": nl * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "errors_vs_oracle": errors,
            "other_workloads": others,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--softcap", type=float, default=0.0,
                    help="--kernel prefill only: the prefill with this SoftCap (profiling "
                         "captures of the capped variant; 0 = none)")
    ap.add_argument("--rms-form", choices=["auto", "fused", "two_pass"], default=None,
                    help="--kernel rmsnorm: call the workspace entry with this form "
                         "(default: the single fused kernel)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the secondary GQA sweep / long-decode measurements")
    ap.add_argument("--kernel", choices=["all", "prefill", "decode", "rmsnorm", "backward"],
                    default="all",
                    help="time the whole step (default) or one kernel only (profiling)")
    ap.add_argument("--batch", type=int, default=16,
                    help="batch rows of the RMSNorm + MatMul workload (--kernel rmsnorm), batch "
                         "of the causal MHA backward (--kernel backward)")
    ap.add_argument("--small", action="store_true",
                    help="decode on a quarter of the batch, prefill on one sequence "
                         "(profiling captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.softcap and (args.kernel != "prefill" or args.impl != "ours"):
        ap.error("--softcap applies to --kernel prefill only")
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel == "rmsnorm":
        return run_rmsnorm(args)
    if args.kernel == "backward":
        return run_backward(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
