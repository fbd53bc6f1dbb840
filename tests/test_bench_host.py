"""Host-side checks of the bench: work accounting pinned to the numbers the
CMU 15-779 第 11 讲 page prints (§1.2, 练习 6; fixture tests/golden/
traffic_model.json), brute-force causal pair counts, and the max/sum over
ranks used for N > 1 (gloo, world size 2, CPU)."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "traffic_model.json")


def test_single_head_traffic_model_matches_lecture():
    g = json.load(open(GOLDEN))["single_head"]
    N, d, e = g["N"], g["d"], g["elem_bytes"]
    # score matrix written once and read once: "67 MB"
    assert round(bench.score_round_trip_bytes(N, e) / 1e6) == g["score_round_trip_MB"]
    # fused I/O of one head (Q, K, V read, O written): "4.2 MB"
    assert round(bench.prefill_io_bytes(1, 1, 1, N, N, d, e) / 1e6, 1) == g["flash_io_MB"]
    # two matmuls, non-causal: "8.6 GFLOP"
    assert round(bench.prefill_flops(1, 1, N, N, d, causal=False) / 1e9, 1) == g["two_matmul_GFLOP"]


def test_gqa_decode_traffic_matches_exercise():
    g = json.load(open(GOLDEN))["gqa_decode"]
    lens = [g["ctx"]] * g["batch"]
    kv = bench.decode_kv_bytes(g["kv_heads"], lens, g["d"], g["elem_bytes"])
    per_q = bench.decode_kv_bytes_per_query_head(g["kv_heads"] * g["group"], lens, g["d"],
                                                 g["elem_bytes"])
    assert round(kv / 1e6) == g["kv_MB"]
    assert round(per_q / 1e6) == g["per_query_head_MB"]
    assert round(per_q / (g["hbm_TBps"] * 1e12) * 1e6) == g["per_query_head_us"]
    assert round(kv / (g["hbm_TBps"] * 1e12) * 1e6) == g["grouped_us"]


@pytest.mark.parametrize("Lq,Lk", [(1, 1), (5, 5), (7, 12), (12, 7), (1, 100), (100, 1),
                                   (4096, 4096), (300, 333)])
def test_causal_pairs_brute_force(Lq, Lk):
    n = sum(1 for i in range(Lq) for j in range(Lk) if j <= i + Lk - Lq)
    assert bench.causal_pairs(Lq, Lk) == n


def test_causal_mha_workload_flops():
    # 4 * 128 * 4 * 32 * 4096 * 4097 / 2
    assert bench.prefill_flops(4, 32, 4096, 4096, 128, True) == 4 * 128 * 4 * 32 * (4096 * 4097 // 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mx = bench.max_over_ranks(float(rank + 1) * 1.5, world)
    sm = bench.sum_over_ranks(float(rank + 1), world)
    q.put((rank, mx, sm))
    dist.destroy_process_group()


def test_max_and_sum_over_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert all(p.exitcode == 0 for p in procs)
    assert [r[1] for r in res] == [3.0, 3.0]
    assert [r[2] for r in res] == [3.0, 3.0]


def test_reference_arm_nonzero_rank_exits_quietly(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_contract_line(monkeypatch, capsys):
    monkeypatch.setattr(bench, "oracle_prefill_sample", lambda budget, seed=0: (2e9, 0.5, "s"))
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip())
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["impl"] == "reference"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert abs(line["value"] - 2e9 / 0.5 / 1e12) < 1e-12


def test_clock_summary_keeps_only_samples_inside_the_region():
    lines = [
        "2026/12/02 07:00:00.000, 0, 2070, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 07:00:01.000, 0, 1500, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 07:00:01.100, 0, 1480, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 07:00:03.000, 0, 2070, 2070, 140.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    t0 = bench.ClockSampler._epoch("2026/12/02 07:00:00.900")
    t1 = bench.ClockSampler._epoch("2026/12/02 07:00:01.200")
    c = bench.ClockSampler.summarize(lines, t0, t1)
    assert c["samples_in_region"] == 2 and c["sm_mhz"] == 1490.0
    assert c["reasons"] == ["sw_power_cap"] and c["sm_max_mhz"] == 2070.0


def test_backward_flops_are_two_and_a_half_forward():
    assert bench.backward_flops(2, 3, 100, 130, 64, True) * 2 == \
        5 * bench.prefill_flops(2, 3, 100, 130, 64, True)


def test_rmsnorm_matmul_traffic_is_the_weight_at_small_batch():
    """Mirage §3.3: at small batch the fused kernel is bound by reading the
    32 MB weight of the LLaMA-2-7B shape (H = D = 4096, bf16)."""
    b = bench.rmsnorm_matmul_bytes(1, 4096, 4096)
    assert 32 * 2 ** 20 <= b <= 32 * 2 ** 20 + 64 * 1024
    assert bench.rmsnorm_matmul_flops(256, 4096, 4096) == 2 * 256 * 4096 * 4096


@pytest.mark.parametrize("Lq,Lk,left,right,causal", [
    (7, 7, 2, -1, True), (7, 9, 3, 1, False), (9, 5, -1, 2, False), (6, 6, -1, -1, True),
    (5, 8, 0, 0, False), (8, 8, 10, -1, True)])
def test_window_pairs_brute_force(Lq, Lk, left, right, causal):
    n = 0
    for i in range(Lq):
        ia = i + Lk - Lq
        for j in range(Lk):
            ok = (left < 0 or j >= ia - left) and (right < 0 or j <= ia + right)
            if causal:
                ok = ok and j <= ia
            n += ok
    assert bench.window_pairs(Lq, Lk, left, right, causal) == n
    if left < 0 and right < 0 and causal:
        assert n == bench.causal_pairs(Lq, Lk)


def test_nvml_summary_keeps_samples_inside_the_region():
    import bench
    samples = [(0.9, 1500.0, 300.0, 0x1), (1.0, 2070.0, 900.0, 0x0),
               (1.1, 2000.0, 1000.0, 0x4), (1.2, 2070.0, 950.0, 0x0), (1.5, 1200.0, 200.0, 0x8)]
    c = bench.NvmlSampler.summarize(samples, 2070.0, 1.0, 1.2)
    assert c["samples_in_region"] == 3 and c["samples"] == 5
    assert c["sm_mhz"] == 2070.0 and c["sm_mhz_min"] == 2000.0
    assert c["reasons"] == ["sw_power_cap"]          # the hw_slowdown sample lies outside
    assert c["power_w_max"] == 1000.0


def test_error_stats_flag_nonzero_rows_that_see_no_key():
    import numpy as np
    import bench
    e = bench.ErrorStats()
    ref = np.zeros((3, 4))
    lr = np.array([-np.inf, 0.5, 1.0])
    got = ref.copy()
    got[1] += 0.01
    e.add("w", got, ref, lr + np.array([0.0, 2e-4, 0.0]), lr)
    s = e.summary()["w"]
    assert abs(s["o_max_abs"] - 0.01) < 1e-12 and abs(s["lse_max_abs"] - 2e-4) < 1e-12
    assert s["empty_rows_exact"]
    got[0, 2] = 1e-3
    e.add("w", got, ref, lr, lr)
    assert not e.summary()["w"]["empty_rows_exact"]
