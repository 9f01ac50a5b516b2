"""Host-side logic of bench.py: the multi-rank timing reduction (gloo,
world_size 2, on CPU), clock parsing, the traffic record guard."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    assert (r, w) == (rank, world)
    bench.barrier(world)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    out[rank] = m
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert out[0] == out[1] == 15.0


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_summarize_clocks():
    lines = ["0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1905, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active",
             "garbage"]
    c = bench.summarize_clocks(lines)
    assert c["samples"] == 2 and c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == 1935.0 and c["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks([])["samples"] == 0


def test_traffic_record_requires_matching_source(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"kern": {"wl": {"source_digest": bench.source_digest([str(src)]), "dram_bytes_per_launch": 123.0}}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("kern", "wl", [str(src)]) == 123.0
    src.write_text("kernel v2")
    assert bench.kernel_traffic("kern", "wl", [str(src)]) is None


def test_byte_and_flop_constants():
    assert bench.STEP_BYTES == 34560
    assert bench.PREFILL_BYTES_PER_TOKEN_HEAD == 1152
    assert bench.PREFILL_FLOP_PER_TOKEN_HEAD == 106496


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_summarize_nvml_reasons_and_median():
    bits = bench.NvmlClockSampler.REASONS
    samples = [(2070, 2070, 0), (2055, 2070, 0x4), (1995, 2070, 0x4 | 0x1), (2070, 2070, 0x40)]
    c = bench.summarize_nvml(samples, bits)
    assert c["samples"] == 4 and c["sm_max_mhz"] == 2070 and c["source"] == "nvml"
    assert c["sm_mhz"] == (2055 + 2070) / 2
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]  # the idle bit (0x1) is not a throttle
    assert bench.summarize_nvml([], bits)["samples"] == 0


def test_oracle_rate_repeats_when_the_units_run_out():
    calls = []

    def fn(n, threads):
        calls.append(n)
        import time
        time.sleep(0.002 * n)

    rate, n, dt = bench.oracle_rate(fn, units=3, budget_s=0.05, threads=1)
    # 3 units take ~6 ms < 50 ms: the full run is repeated until the budget is spent
    assert n % 3 == 0 and n >= 6 and dt >= 0.04
    assert abs(rate - n / dt) < 1e-9


def test_oracle_rate_grows_the_sample_to_the_budget():
    def fn(n, threads):
        import time
        time.sleep(0.001 * n)

    rate, n, dt = bench.oracle_rate(fn, units=10 ** 6, budget_s=0.03, threads=4)
    assert dt >= 0.03 and n < 10 ** 6


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line
    with the contract's keys, its own cpu_baseline and an e2e with no copies."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_committed_traffic_records_match_the_kernel_sources():
    """The DRAM traffic the bench reports comes from the committed ncu record only while
    the kernel's sources are unchanged; the records in profiles/traffic.json must name
    the current sources (re-capture, or restate an unchanged kernel's digest, after an
    edit)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    csrc = os.path.join(root, "rwkv_linear_attention_gb300", "csrc")
    shared = [os.path.join(csrc, "sm103_ptx.cuh"), os.path.join(csrc, "wkv7_internal.cuh")]
    sources = {"wkv7_step_kernel": "wkv7_step.cu", "wkv7_prefill_chunked_kernel": "wkv7_prefill_chunked.cu",
               "bwd_grad_tc_kernel": "wkv7_prefill_backward.cu", "bwd_summary_tc_kernel": "wkv7_prefill_backward.cu"}
    with open(os.path.join(root, "profiles", "traffic.json")) as f:
        records = json.load(f)
    for kernel, src in sources.items():
        digest = bench.source_digest([os.path.join(csrc, src)] + shared)
        assert kernel in records, kernel
        for workload, rec in records[kernel].items():
            assert rec["source_digest"] == digest, f"{kernel} / {workload}: record is for other sources"
            assert rec["dram_bytes_per_launch"] == rec["read_bytes"] + rec["write_bytes"]
