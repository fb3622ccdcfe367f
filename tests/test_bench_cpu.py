"""Host-side logic of bench.py: the reference arm's JSON line, the clock
summary, the profile lookup, and the max-over-ranks timing of the replica
mode (two gloo ranks on CPU)."""

import contextlib
import io
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_reference_arm_json_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1", "--ref-rows", "4"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["warmup"] == 3          # at least three warm-up steps
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_grpo_json_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--path", "grpo", "--grpo-n", "65536", "--grpo-seqs", "64",
                    "--steps", "1", "--warmup", "1", "--ref-rows", "2"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["config"]["tokens_per_step"] == 16384 and line["cpu_baseline"]["kind"] == "oracle"


def test_clock_summary_parsing():
    s = bench.ClockSampler(0)
    s.out = ("2026/12/02 10:00:00.100, 0, 1500, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "2026/12/02 10:00:00.300, 0, 1980, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
             "2026/12/02 10:00:00.500, 0, 1990, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "2026/12/02 10:00:00.700, 0, 2000, 2070, 980.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "2026/12/02 10:00:00.900, 0, 900, 2070, 200.5, 0x0, Not Active, Active, Not Active, Not Active\n")
    c = s.summary()                      # no window marked: every sample
    assert c["samples"] == 5 and "hw_thermal_slowdown" in c["reasons"]
    t = bench.ClockSampler._stamp
    s.window = (t("2026/12/02 10:00:00.250"), t("2026/12/02 10:00:00.750"))
    c = s.summary()                      # only the samples inside the timed region
    assert c["sm_mhz"] == 1990 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    s.window = None
    s.mark()
    s.mark()
    assert s.window[0] <= s.window[1]
    s.out = ""
    assert s.summary()["reasons"] == ["unavailable"]


def test_profiled_traffic_requires_current_kernel_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (tmp_path / "selected_token_logprob_gb300" / "csrc").mkdir(parents=True)
    for fn in ("logp_kernels.cuh", "logp_prims.cuh"):
        src = os.path.join(bench.ROOT, "selected_token_logprob_gb300", "csrc", fn)
        (tmp_path / "selected_token_logprob_gb300" / "csrc" / fn).write_bytes(open(src, "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench._kernel_hash()
    (prof / "k_logp_bwd_long.md").write_text(
        f"kernel_source_sha256_16: {h}\ndram_bytes_per_launch: 1.99e10\n")
    assert bench._profiled_traffic("k_logp_bwd") == pytest.approx(1.99e10)
    (prof / "k_logp_bwd_long.md").write_text(
        "kernel_source_sha256_16: 0000000000000000\ndram_bytes_per_launch: 1.99e10\n")
    assert bench._profiled_traffic("k_logp_bwd") is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench._max_over_ranks(10.0 + rank, world, torch.device("cpu"))
        bench._barrier(world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}
