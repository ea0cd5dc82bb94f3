"""The multi-rank parts of bench.py on CPU, with two gloo ranks: the slowest
rank's time is what every rank reports, whole-job throughput counts every
rank's tokens, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_max = bench.max_over_ranks(times[rank])
        out[rank] = (ms_max, bench.whole_job_tokens_per_s(64, world, ms_max * 1e-3))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_all_tokens():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        times = [1.5, 2.5]
        mp.start_processes(_rank_main, args=(2, _free_port(), times, out), nprocs=2, start_method="spawn")
        got = dict(out)
    assert got[0][0] == got[1][0] == 2.5
    assert got[0][1] == got[1][1] == pytest.approx(2 * 64 / 2.5e-3)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_tokens_per_s(64, 1, 2e-3) == pytest.approx(32000.0)


def test_reference_arm_prints_nothing_off_rank_0(monkeypatch, capsys):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(argparse.Namespace(workload="tiny", steps=2, warmup=1, gpus=2))
    assert capsys.readouterr().out == ""


def test_kernel_roofline_takes_the_slower_roof():
    import bench
    hbm, tc = 6788.6, 1722.1
    # a decode-shaped gate/up launch: 291 experts' weights, 512 rows -> bytes dominate
    dec = bench.kernel_roofline("gemm_gate_up", 4.815e9, 2.0 * 512 * 7168 * 4096, 1.1, None, hbm, tc, "measured")
    assert dec["bound"] == "hbm" and dec["unit"] == "GB/s"
    assert dec["frac"] == pytest.approx(4.815e9 / 1.1e-3 / 1e9 / hbm)
    # a prefill-shaped one: 32768 rows over 384 experts -> flops dominate
    fl = 2.0 * 32768 * 7168 * 4096
    pre = bench.kernel_roofline("gemm_gate_up", 6.946e9, fl, 2.72, None, hbm, tc, "measured")
    assert pre["bound"] == "tensor" and pre["unit"] == "TFLOP/s" and pre["peak"] == tc
    assert pre["frac"] == pytest.approx(fl / 2.72e-3 / 1e12 / tc)


def test_profile_traffic_only_for_the_captured_source(monkeypatch, tmp_path):
    """`roofline.traffic` comes from a committed ncu summary only while the kernel source still
    hashes to the one the summary was captured from."""
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.kernel_source_sha()
    (prof / "gemm_gate_up_w1.md").write_text(f"source_sha256: {sha}\ndram_bytes_per_launch: 4.8e9\n")
    (prof / "gemm_gate_up_w2.md").write_text(f"source_sha256: {'0' * 64}\ndram_bytes_per_launch: 4.8e9\n")
    (prof / "gemm_gate_up_w3.md").write_text(f"source_sha256: {sha}\n")
    real_root = bench.ROOT
    csrc = tmp_path / "w4a16_mixture_experts_sigmoid_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        (csrc / f).write_bytes(open(f"{real_root}/w4a16_mixture_experts_sigmoid_gb300/csrc/{f}", "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("gemm_gate_up", "w1") == 4.8e9
    assert bench.profile_traffic("gemm_gate_up", "w2") is None       # another kernel source
    assert bench.profile_traffic("gemm_gate_up", "w3") is None       # no byte count
    assert bench.profile_traffic("gemm_gate_up", "absent") is None
