"""bench.py's multi-process host logic on CPU: two gloo ranks, no GPU.

Each rank of `bench.py --gpus N` runs an independent replica (the decode path has
no exchange step); rank 0 reports all ranks' work over the slowest rank's time.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._rank_env() == (rank, world, rank)
        t = bench.slowest_rank_ms(times[rank], dist)
        value, tmax = bench.aggregate([t] * world, [1000] * world)
        out.put((rank, t, value, tmax))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    times = [12.5, 20.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(out.get(timeout=10) for _ in range(2))
    for rank, t, value, tmax in got:
        assert t == 20.0 and tmax == 20.0
        # 2 ranks x 1000 units over the slowest rank's 20 ms
        assert value == pytest.approx(2000 / 0.020)


def _reference_rank(rank, world, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    out.put((rank, bench.main(["--impl", "reference", "--gpus", str(world),
                               "--steps", "1", "--warmup", "3"])))


def test_reference_arm_other_ranks_exit_without_work():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    p = ctx.Process(target=_reference_rank, args=(1, 2, out))
    p.start()
    p.join(timeout=60)
    assert p.exitcode == 0
    assert out.get(timeout=10) == (1, 0)


def test_roofline_bound_follows_the_longer_time():
    """The long-context call is HBM-bound, the 4-draft speculative call tensor-bound
    (at the fp8 peak), from the algorithmic bytes and flops of the workloads."""
    import bench
    from paged_mla_decode_gb300 import accounting
    from paged_mla_decode_gb300 import workloads as wl

    hbm, _ = bench.measured_peaks()
    fp8, _ = bench.tensor_peak("fp8")
    bf16, _ = bench.tensor_peak("bf16")
    assert fp8 == 2 * bf16
    for make, bound in ((wl.long_context, "hbm"), (wl.speculative, "tensor")):
        w = make()
        nbytes = accounting.step_bytes(w.seq_lens, w.num_queries, w.num_heads, "e4m3",
                                       unique_tokens=w.unique_tokens)["total"]
        flops = accounting.step_flops(w.seq_lens, w.num_queries, w.num_heads)
        first, other = bench.rooflines(nbytes, flops, 100.0, hbm, "m", fp8, "m")
        assert first["bound"] == bound and other["bound"] != bound
        # achieved = algorithmic work / time; frac = achieved / peak
        assert abs(first["frac"] - first["achieved"] / first["peak"]) < 1e-12
    # a call that takes exactly the HBM time at peak reads 1.0 of the HBM roofline
    first, _ = bench.rooflines(6.76e9, 1.0, 1000.0, 6760.0, "m", fp8, "m")
    assert first["bound"] == "hbm" and abs(first["frac"] - 1.0) < 1e-9


def test_reference_arm_line_has_the_contract_keys(capsys, monkeypatch):
    """`bench.py --impl reference` (the float64 oracle on the host cores) prints one
    JSON line with the keys the driver reads; checked on the tiny workload."""
    import json

    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1",
                       "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_clock_record_keeps_this_gpus_rows():
    """The clock sampler keeps the rows of the GPU whose UUID torch reports.

    nvidia-smi prints UUIDs as GPU-<uuid>; torch may give the bare UUID: both
    spellings select the same rows, and a lone GPU is kept even without a match.
    """
    text = "\n".join([
        "GPU-aaaa-1, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "GPU-bbbb-2, 1200, 2070, 300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "GPU-aaaa-1, 2050, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "GPU-aaaa-1, 2070, 2070, 980.0, 0x4, Not Active, Not Active, Not Active, Active",
    ])
    sys.path.insert(0, ROOT)
    import bench
    rec = bench.ClockSampler.summarise(text, "aaaa-1")
    assert rec["samples"] == 3 and rec["sm_mhz"] == 2070 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler.summarise(text, bench._norm_uuid("GPU-AAAA-1")) == rec
    lone = "\n".join(l for l in text.splitlines() if "bbbb" in l)
    assert bench.ClockSampler.summarise(lone, "cccc")["sm_mhz"] == 1200
    assert bench.ClockSampler.summarise(text, "cccc") is None
