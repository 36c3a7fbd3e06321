"""Host-side pieces of bench.py, on CPU: the algorithmic bytes per decode token (the roofline's
numerator) against the per-config figures computed independently for the hot-path scope table,
and the multi-replica timing (max over ranks, whole-job throughput) on two `gloo` ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


@pytest.mark.parametrize("name,ctx,weights_gb,kv_mb", [
    ("llama3_8b", 8192, 7.974, 2147.5),
    ("qwen3_0_6b", 128, 1.192, 29.4),
    ("qwen3_0_6b", 1024, 1.192, 234.9),
    ("qwen3_0_6b", 4096, 1.192, 939.5),
    ("qwen2_7b", 2048, 3.977, 234.9),
    ("gemma3_1b", 8192, 2.000, 90.2),   # 22 of 26 layers see their last 512 keys
])
def test_decode_bytes_per_token_match_the_scope_table(name, ctx, weights_gb, kv_mb):
    total, w, kv = bench.decode_bytes_per_token(synth.CONFIGS[name], ctx)
    assert abs(w / 1e9 - weights_gb) <= 0.002          # row padding to 32 bytes adds < 0.02 %
    assert abs(kv / 1e6 - kv_mb) <= 0.05
    assert total == w + kv


def test_f16_cache_halves_the_kv_bytes_only():
    cfg = synth.CONFIGS["llama3_8b"]
    t32, w32, kv32 = bench.decode_bytes_per_token(cfg, 8192)
    t16, w16, kv16 = bench.decode_bytes_per_token(cfg, 8192, kv_elt=2)
    assert w16 == w32 and kv16 == kv32 / 2


def test_single_rank_timing_is_the_rank_time():
    assert bench.max_over_ranks(12.5, 1, torch, "cpu") == 12.5
    assert bench.job_throughput(512, 1, 1000.0) == 512.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, torch, "cpu")
        out.put((rank, ms, bench.job_throughput(100, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_summed_tokens():
    """Replicas only: no collective on the data path, but the timed region's time is the maximum
    over ranks and the job's tokens/s counts every replica's tokens."""
    world, times = 2, [40.0, 50.0]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tps in res:
        assert ms == 50.0
        assert tps == pytest.approx(100 * world / 0.050)


def test_reference_arm_on_a_non_zero_rank_does_no_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    # rank 1 returns before it reads its arguments, imports the oracle or builds any model
    assert bench.run_reference(None) is None


def test_host_cpu_names_the_architecture_and_core_count():
    import platform
    s = bench.host_cpu()
    assert platform.machine() in s and f"{os.cpu_count()} logical cores" in s


def test_host_cpu_names_an_arm_server_core_from_its_part_number(monkeypatch):
    import builtins
    import io
    real_open = builtins.open
    text = "processor\t: 0\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n\nprocessor\t: 1\nCPU implementer\t: 0x41\n"
    monkeypatch.setattr(builtins, "open", lambda f, *a, **k: io.StringIO(text) if f == "/proc/cpuinfo"
                        else real_open(f, *a, **k))
    assert bench.host_cpu().startswith("Arm Neoverse-V2 (")


def test_in_step_roofline_divides_the_kinds_bytes_by_its_share_of_the_timed_step():
    prof = {"gemv": {"launches": 64, "ms": 6.0, "bytes": 8e9, "flops": 0.0},
            "attention": {"launches": 16, "ms": 2.0, "bytes": 1e9, "flops": 0.0}}
    r = bench.in_step_roofline(prof, 16, 2.0, 6800.0)
    # share 0.75 of a 2 ms step: 1.5 ms for 0.5 GB per step -> 333.3 GB/s
    assert abs(r["share_of_step"] - 0.75) < 1e-12
    assert abs(r["ms_per_step"] - 1.5) < 1e-12
    assert abs(r["achieved"] - 0.5e9 / 1.5e-3 / 1e9) < 1e-6
    assert abs(r["us_per_launch"] - 1500.0 / 4) < 1e-9
    assert r["achieved"] * r["ms_per_step"] / 1000.0 <= r["bytes_per_step"] / 1e9 * 1.0000001
    assert bench.in_step_roofline(prof, 16, 2.0, 6800.0, kind="argmax") is None


@pytest.mark.parametrize("name,ctx", sorted(bench.TARGET_70))
def test_decode_targets_are_70_percent_of_8_tbs_at_the_workloads_bytes(name, ctx):
    bpt, _, _ = bench.decode_bytes_per_token(synth.CONFIGS[name], ctx)
    assert abs(bench.TARGET_70[(name, ctx)] - 0.7 * 8e12 / bpt) / bench.TARGET_70[(name, ctx)] < 0.01
