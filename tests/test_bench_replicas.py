"""The N > 1 bookkeeping of bench.py, on two gloo ranks on CPU.

Multi-GPU here is replicas only: every rank runs its own copy of the
workload, with no collective on the data path.  What N > 1 changes is the
reporting: the job's step time is the slowest rank's (a max-reduction after
a barrier), the throughput counts the work of every rank, and the reference
arm runs on rank 0 alone."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    step_ms = 1.5 * (rank + 1)  # rank r took 1.5 * (r + 1) ms per step
    slowest = bench.max_over_ranks(step_ms, world, "cpu")
    value = bench.replica_throughput(world, 2e12, slowest)  # 2 TFLOP per step per replica
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "value": value}, f)


def test_two_gloo_ranks_take_the_slowest_rank_and_count_both(tmp_path):
    import torch.multiprocessing as mp
    mp.start_processes(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    r = [json.load(open(tmp_path / f"r{k}.json")) for k in range(2)]
    assert r[0]["slowest"] == r[1]["slowest"] == 3.0
    assert r[0]["value"] == pytest.approx(2 * 2e12 / 3.0e-3 / 1e12)
    assert r[1]["value"] == r[0]["value"]


def test_one_rank_reports_its_own_time():
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.replica_throughput(1, 1e12, 1.0) == pytest.approx(1000.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload = bench.DEFAULT_WORKLOAD
        steps = 1
        warmup = 0

    bench.run_reference(Args())
    assert capsys.readouterr().out == ""


def test_delayed_scaling_mode_plan():
    """--modes per_tensor_static: per linear the static activation quantize
    (two launches: zeroing kernel + cast), the weight quantize, the GEMM and
    the scale update; the algorithmic bytes count one read of A, one write
    of q, the scale read and the amax write."""
    import bench

    class Args:
        workload = "tinyllama_1.1b_m512"
        modes = "per_tensor_static"

    wl = bench.workload_of(Args())
    assert wl.modes == ("per_tensor_static",)
    plan = bench.kernel_plan(wl)
    assert len(plan) == len(wl.linears)
    for lin, mode, ks in plan:
        names = [k[0] for k in ks]
        assert names == ["quant_static_act", "quant_per_tensor_weight", "gemm_per_tensor", "scale_from_history"]
        assert ks[0][2] == lin.M * lin.K * 3 + 8
        assert ks[3][2] == 4 * bench.HIST_LEN + 4
        assert ks[2][3] == 2 * lin.M * lin.N * lin.K


def test_unknown_mode_is_rejected():
    import bench

    class Args:
        workload = "tinyllama_1.1b_m512"
        modes = "per_tensor,bogus"

    with pytest.raises(SystemExit):
        bench.workload_of(Args())


def test_per_channel_mode_plan():
    import bench

    class Args:
        workload = "llama2_7b_m128"
        modes = "per_channel"

    plan = bench.kernel_plan(bench.workload_of(Args()))
    for lin, mode, ks in plan:
        assert [k[0] for k in ks] == ["quant_per_tensor_act", "quant_per_channel_weight", "gemm_per_channel"]
        assert ks[1][2] == lin.N * lin.K * 3 + 4 * lin.N
        assert ks[2][2] == lin.M * lin.K + lin.N * lin.K + 4 + 4 * lin.N + 2 * lin.M * lin.N


def test_both_arms_print_the_same_config():
    """The GPU arm and the reference arm build `config` with one helper, so
    the two lines name the same workload in the same words."""
    import bench

    class Args:
        workload = bench.DEFAULT_WORKLOAD
        modes = ""
        gpus = 1

    wl = bench.workload_of(Args())
    cfg = bench.config_of(Args(), wl)
    assert cfg["workload"] == "outlier_16384x8192x8192"
    assert cfg["linears"] == [["gemm", 16384, 8192, 8192]]
    assert set(cfg) == {"workload", "description", "linears", "modes", "in_dtype", "out_dtype", "l2", "parallelism"}


def test_reference_arm_line(monkeypatch, capsys):
    """On rank 0 the reference arm prints one line with the shared config,
    a cpu_baseline describing its own sample and an e2e of zero copies."""
    import json

    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class Args:
        workload = "per_tensor_64x64x128"
        modes = ""
        gpus = 1
        steps = 2
        warmup = 1

    bench.run_reference(Args())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.config_of(Args(), bench.workload_of(Args()))
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["samples"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_oracle_sample_is_fixed():
    """Both arms time the same sample: the GEMM rows depend on the workload only."""
    import bench
    import synth
    wl = synth.WORKLOADS["outlier_16384x8192x8192"]
    assert bench.oracle_sample_rows(wl) == bench.oracle_sample_rows(wl) == [149]
    wl = synth.WORKLOADS["llama2_7b_m1"]
    assert bench.oracle_sample_rows(wl) == [1, 1, 1, 1]


def test_default_lines_end_with_the_headline():
    """A plain run prints the decode (unfused vs fused) and UE8M0 lines first
    and the largest block-scaled workload last."""
    import bench

    class Args:
        workload = None
        modes = ""
        gpus = 1

    lines = bench.lines_of(Args())
    assert [(a.workload, a.modes) for a in lines][-1] == ("outlier_16384x8192x8192", "")
    assert ("llama2_7b_m1", "block_fp8w,fused_fp8w") in [(a.workload, a.modes) for a in lines]
    Args.workload = "llama2_7b_m8"
    assert [(a.workload, a.modes) for a in bench.lines_of(Args())] == [("llama2_7b_m8", "")]


def test_fused_and_ue8m0_plans():
    import bench

    class Args:
        workload = "llama2_7b_m1"
        modes = "block,fused,block_ue8m0"

    plan = bench.kernel_plan(bench.workload_of(Args()))
    names = {mode: [k[0] for k in ks] for lin, mode, ks in plan if lin.name == "o"}
    assert names["fused"] == ["quant_weight_block", "linear_fused"]
    assert names["block_ue8m0"] == ["quant_token_group_ue8m0", "quant_weight_block_ue8m0", "gemm_block_ue8m0"]
    fused = [ks for lin, mode, ks in plan if lin.name == "o" and mode == "fused"][0]
    M, N, K = 1, 4096, 4096
    assert fused[1][2] == M * K * 2 + N * K + 4 * 32 * 32 + 2 * M * N and fused[1][3] == 2 * M * N * K


def test_fp8_weight_plans():
    """Weights held in FP8: a step is the activation quantize + GEMM, or the
    fused linear alone; no weight quantization in the step."""
    import bench

    class Args:
        workload = "llama2_7b_m1"
        modes = "block_fp8w,fused_fp8w"

    plan = bench.kernel_plan(bench.workload_of(Args()))
    for lin, mode, ks in plan:
        names = [k[0] for k in ks]
        assert "quant_weight_block" not in names
        assert names == (["quant_token_group", "gemm_block"] if mode == "block_fp8w" else ["linear_fused"])
