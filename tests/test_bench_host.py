"""Host-side logic of bench.py: byte model, clock-log parsing, and the
max-over-ranks aggregation of the replica runs (2 gloo ranks on CPU)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from synth import get_preset


def test_step_bytes_of_bench_workload():
    run = get_preset("gpt2m_q4")
    mb = bench.mean_step_bytes(run.model, run.prompt_len, run.n_steps) / 1e6
    # 173.6 MB of Q4_0 weights + 27.1 MB mean KV read over positions 150..399 + small tensors
    assert 201.5 < mb < 202.5
    q8 = get_preset("gpt2m_q8")
    assert 355.5 < bench.mean_step_bytes(q8.model, 150, 250) / 1e6 < 357.5


def test_step_bytes_of_the_other_formats():
    """Q5_0 streams 22/18 of Q4_0's weight bytes; a 4-bit group-64 code predictor
    replaces 68/64 by 36/64 bytes per weight on the code predictor's share only."""
    q4, q5 = get_preset("gpt2m_q4"), get_preset("gpt2m_q5")
    w4 = q4.model.quantised_params_per_step() * 18 / 32
    d = bench.step_bytes(q5.model, 200) - bench.step_bytes(q4.model, 200)
    assert abs(d - w4 * (22 / 18 - 1)) < 16
    a8, cp4 = get_preset("qwen_a8"), get_preset("qwen_a8_cp4")
    cp_params = a8.model.quantised_params_per_step() - a8.model.talker_params()
    d = bench.step_bytes(a8.model, 300) - bench.step_bytes(cp4.model, 300)
    assert abs(d - cp_params * (68 - 36) / 64) < 16
    # the printed code-predictor traffic of the 8-bit frame ([B] section 3: 1.29 GB) halves, about
    assert 0.6e9 < cp_params * 36 / 64 < 0.7e9


def test_clock_summary_parsing(tmp_path):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "c.csv")
    with open(cs.path, "w") as f:
        f.write("0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1980, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1995, 2070, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    s = cs.summary()
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    d = bench.init_dist(ws, "gloo")
    bench.barrier(d, ws)
    t = bench.max_over_ranks(d, ws, 1.0 + rank)       # rank 1 is the slowest
    out[rank] = t
    d.destroy_process_group()


def test_max_over_ranks_gloo():
    ws = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(ws, _free_port(), out), nprocs=ws, join=True)
    assert out[0] == out[1] == 2.0


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""
