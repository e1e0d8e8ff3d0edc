"""Host-side logic of bench.py (CPU only): clock parsing, max over ranks with a
2-rank gloo group, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_summarize_clocks():
    text = ("0, 1890, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active\n"
            "0, 1905, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            "0, 165, 2070, 120.0, 0x1, Not Active, Not Active, Not Active, Not Active\n"
            "garbage line\n")
    c = bench.summarize_clocks(text)
    assert c["sm_max_mhz"] == 2070.0
    assert c["samples"] == 2                      # idle sample (120 W) excluded
    assert c["sm_mhz"] in (1890.0, 1905.0)
    assert c["reasons"] == ["sw_power_cap"]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.max_over_ranks(10.0 + rank * 5.0, world, device="cpu")
    bench.barrier(world)
    out[rank] = v
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 15.0 and out[1] == 15.0


def test_single_rank_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_flop_accounting():
    assert bench.mlp_flop() == 12 * 4096 * 3072 * 12288
    assert bench.ce_flop() == 2 * 8192 * 1536 * 51200
    assert bench.step_flop() == bench.mlp_flop() + bench.ce_flop()


def test_physical_gpu(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.physical_gpu(1) == "5"
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.physical_gpu(0) == "0"


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU-only check of the reference arm's line")
def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["metric"] == bench.METRIC


def test_combine_row_bytes():
    # The combine reads the (max, sum-exp) planes of every partition (2 P T floats), the
    # target and one target logit per token, and writes the loss: 8 P T + 12 T bytes.
    import tensor_transformer_layer_gb300 as mp
    T = bench.CE["T"]
    P = mp.mp_vocab_ce_workspace_bytes(T, bench.CE["v_pad"], bench.CE["t"]) // (12 * T)
    assert P * 12 * T == mp.mp_vocab_ce_workspace_bytes(T, bench.CE["v_pad"], bench.CE["t"])
    row = bench.combine_row(0.01, {"hbm_gbs": 5000.0}, "test")
    assert row["bytes"] == 8 * P * T + 12 * T and row["partitions"] == P
    assert abs(row["achieved_gbs"] - row["bytes"] / 1e-5 / 1e9) < 1e-6
    assert abs(row["frac"] - row["achieved_gbs"] / 5000.0) < 1e-12 and row["bound"] == "hbm"


def test_clock_rows_with_timestamps_and_binning():
    import datetime
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)
    lines = []
    for i, mhz in enumerate((1600, 1610, 1900, 1905, 1898)):
        ts = (base + datetime.timedelta(milliseconds=100 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append(f"{ts}, 0, {mhz}, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active")
    text = "\n".join(lines) + "\n"
    rows = bench.parse_clock_rows(text, timestamps=True)
    assert len(rows) == 5 and rows[0][1] == 1600.0 and rows[1][0] - rows[0][0] == pytest.approx(0.1, abs=1e-6)
    c = bench.summarize_clocks(text, timestamps=True)
    assert c["samples"] == 5 and c["reasons"] == ["sw_power_cap"] and c["sm_mhz"] == 1898.0
    t0 = rows[0][0]
    # chunk 0 covers the two 1.6 GHz samples, chunk 1 the three 1.9 GHz ones, chunk 2 no sample
    windows = [(t0 - 0.01, t0 + 0.15), (t0 + 0.15, t0 + 0.45), (t0 + 1.0, t0 + 2.0)]
    bins = bench.bin_chunks_by_clock(windows, [2.0, 1.0, 1.0], 1e12, rows, bin_mhz=60.0)
    assert [b["chunks"] for b in bins] == [1, 1]
    assert bins[0]["mhz_bin"] == 1620.0 and bins[1]["mhz_bin"] == 1920.0
    assert bins[0]["tflops"] == pytest.approx(1e12 / 2e-3 / 1e12) and bins[1]["tflops"] == pytest.approx(1000.0)


def test_rounded_keeps_structure():
    v = bench.rounded({"a": 1.23456789, "b": [2.0000001, None, "x"], "c": {"d": float("nan"), "e": 0.0}}, 4)
    assert v["a"] == 1.235 and v["b"] == [2.0, None, "x"] and v["c"]["e"] == 0.0 and v["c"]["d"] != v["c"]["d"]
