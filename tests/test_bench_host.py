"""Host-side pieces of bench.py (no GPU needed)."""
import bench


def test_source_fingerprint_ignores_comments_not_code(tmp_path):
    base = "int f(int a) { return a + 1; }  // one\n/* two\n lines */\nint g;\n"
    same = "// header\nint  f(int a)\n{ return a + 1; }\n/* changed */ int g;  // note\n"
    other = "int f(int a) { return a + 2; }\nint g;\n"
    paths = []
    for i, text in enumerate((base, same, other)):
        p = tmp_path / f"k{i}.cuh"
        p.write_text(text)
        paths.append(str(p))
    a, b, c = (bench.source_fingerprint(p) for p in paths)
    assert a == b
    assert a != c


def test_traffic_entry_is_keyed_by_the_code_fingerprint():
    import json
    import os
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    ent = d["gemv_q4_k_b1"]
    assert len(ent["source_fingerprint"]) == 16
    assert ent["dram_bytes_per_launch_avg"] > 0


def _rank_main(rank, world, port, ms_of_rank, out_dir):
    import os
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(ms_of_rank[rank], dist, torch.device("cpu"))
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr(got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_report_the_slowest_rank_and_the_whole_job(tmp_path):
    """world_size 2 over gloo: both ranks see the slower rank's time, and the
    whole-job figure counts both replicas' bytes in that time."""
    import torch.multiprocessing as mp
    ms_of_rank = [3.25, 5.5]
    mp.start_processes(_rank_main, args=(2, _free_port(), ms_of_rank, str(tmp_path)), nprocs=2,
                       start_method="spawn")
    got = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(2)]
    assert got == [5.5, 5.5]
    step_bytes = 3934781440
    assert bench.whole_job_gbs(2, step_bytes, 5.5) == 2 * bench.whole_job_gbs(1, step_bytes, 5.5)
    assert abs(bench.whole_job_gbs(1, step_bytes, 1.0) - step_bytes / 1e6) < 1e-6


def test_single_process_time_is_its_own():
    assert bench.max_over_ranks(4.0, None, None) == 4.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    """Under torchrun only rank 0 runs the oracle arm; the others return 0 at once."""
    import argparse
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.run_reference(argparse.Namespace(steps=1, warmup=3)) == 0


CLOCK_LINES = [
    "2026/12/02 22:30:01.100, 2070, 2070, 900.50, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
    "2026/12/02 22:30:01.300, 1965, 2070, 1395.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
    "garbage line\n",
    "2026/12/02 22:30:01.500, 2070, 2070, 1010.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
    "2026/12/02 22:30:09.000, 1200, 2070, 300.00, 0x0000000000000008, Active, Not Active, Not Active, Not Active\n",
]


def test_clock_lines_parse_and_summarise_over_the_timed_window():
    rows = bench.parse_clock_lines(CLOCK_LINES)
    assert len(rows) == 4                                   # the malformed line is skipped
    assert [r["sm"] for r in rows] == [2070.0, 1965.0, 2070.0, 1200.0]
    t0, t1 = rows[0]["t"], rows[2]["t"]
    assert abs((t1 - t0) - 0.4) < 1e-6
    s = bench.summarise_clocks(rows, t0, t1)
    # the slowdown sample lies outside the timed window; the power cap inside it is kept
    assert s["samples"] == 3 and s["window"] == "timed region"
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    whole = bench.summarise_clocks(rows, rows[0]["t"], rows[3]["t"])
    assert whole["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_summary_without_nvidia_smi():
    s = bench.summarise_clocks([], 0.0, 1.0)
    assert s["samples"] == 0 and s["sm_mhz"] is None


def test_clock_sampler_reads_a_running_sampler(tmp_path, monkeypatch):
    """ClockSampler end to end against a stand-in `nvidia-smi` on PATH that
    prints one sample line every 50 ms until it is stopped."""
    import os
    import sys
    import time
    fake = tmp_path / "nvidia-smi"
    fake.write_text(
        "#!" + sys.executable + "\n"
        "import sys, time\n"
        "while True:\n"
        "    t = time.time()\n"
        "    stamp = time.strftime('%Y/%m/%d %H:%M:%S', time.localtime(t)) + '.%03d' % int((t % 1) * 1000)\n"
        "    print(stamp + ', 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active', flush=True)\n"
        "    time.sleep(0.05)\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ.get("PATH", ""))
    s = bench.ClockSampler(0)
    with s:
        t0 = time.time()
        time.sleep(0.4)
        t1 = time.time()
    rows = s.samples()
    assert len(rows) >= 4 and s.samples() is rows
    summary = bench.summarise_clocks(rows, t0, t1)
    assert summary["sm_mhz"] == 2070.0 and summary["reasons"] == [] and summary["samples"] >= 3


def test_result_line_carries_every_contract_key():
    import argparse
    import json
    r = {"value": 3500.04, "ms_per_step": 1.12207, "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
         "roofline": {"bound": "hbm", "achieved": 3338.0, "peak": 6800.0, "unit": "GB/s", "frac": 0.4909,
                      "traffic": 30754176.0},
         "e2e": {"value": 3443.3, "unit": "GB/s", "h2d_bytes_per_step": 73728, "d2h_bytes_per_step": 16384},
         "gpu_launches": 128000, "extra": {}}
    cpu = {"value": 0.81, "unit": "GB/s", "cores": 16, "kind": "oracle", "sample": "…"}
    line = json.loads(json.dumps(bench.result_line(r, 1, argparse.Namespace(steps=1000, warmup=20), cpu)))
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
              "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 1000 and line["warmup"] == 20
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["data"] == "synthetic" and "workload" in line["config"]
    assert not any(k in line["config"] for k in ("model", "global_batch", "seq_len"))
    assert set(line["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert set(line["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_line(monkeypatch, capsys):
    """The oracle arm on rank 0 prints one line with impl, the contract keys, a
    cpu_baseline describing the run and an e2e without transfers (the oracle
    samples are stubbed here: 1 GB in 2 s a step)."""
    import argparse
    import json
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    calls = []

    def fake_run(orc, synth, frac, threads, seed=2):
        calls.append(frac)
        return 1e9, 2.0
    monkeypatch.setattr(bench, "oracle_sample_run", fake_run)
    assert bench.run_reference(argparse.Namespace(steps=4, warmup=3)) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] == 0.5 and line["unit"] == "GB/s"
    assert line["ms_per_step"] == 2000.0 and line["steps"] == 4 and line["warmup"] == 3
    assert len(calls) == 1 + 3 + 4                          # calibration, warm-up, timed steps
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1 and line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": 0.5, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["metric"] == bench.METRIC and line["config"] == bench.workload_config()
