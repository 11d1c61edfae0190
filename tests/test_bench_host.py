"""Host logic of bench.py on CPU: the max-over-ranks reduction with two gloo
ranks, and the reference arm (the float64 oracle) on rank 0 / other ranks."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    q.put((rank, bench.max_over_ranks([rank + 1.0, 10.0 - rank, 0.5], world, "cpu")))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [2.0, 10.0, 0.5]


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3, 1.5], 1) == [3.0, 1.5]


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                           "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_line_on_rank0():
    r = _run_reference({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_summary_from_nvidia_smi_lines():
    sys.path.insert(0, ROOT)
    import bench

    lines = ["2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "2070, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "truncated, line"]
    c = bench.summarize_clocks(lines)
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = lines[:1] + ["1500, 2070, 1400, 0x48, Not Active, Active, Not Active, Not Active"]
    assert bench.summarize_clocks(hot)["reasons"] == ["hw_thermal_slowdown"]
    assert bench.summarize_clocks([]) is None


def test_linear_launch_count_follows_the_workspace_layout():
    sys.path.insert(0, ROOT)
    import bench

    base = 256 + 8 * 3584 + 8 * 448  # header, codes and scales of 8 x 7168
    assert bench.linear_kernels_per_call(8, 7168, base) == 3
    assert bench.linear_kernels_per_call(8, 7168, base + 8 * 8 * 1536 * 4) == 4
    big = 256 + 4096 * 3584 + 4096 * 448
    assert bench.linear_kernels_per_call(4096, 7168, big) == 4
    assert bench.linear_kernels_per_call(4096, 7168, big + 256) == 5


def test_workload_config_counts_the_routing_and_matches_the_reference_arm():
    """workload_config: active experts, valid slots, the largest load and the
    zero-token experts from per-expert counts; the reference arm's line (run
    on CPU here) carries the config the forward's arm builds from the same
    seeded batch."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    from nvfp4_block_scaled_topk_gb300 import inputs

    cfg = inputs.CONFIGS["tiny"]
    c = bench.workload_config(cfg, np.array([3, 0, 5, 0, 1, 0, 0, 7]), world=2)
    assert (c["active_experts"], c["valid_slots"], c["max_expert_load"], c["zero_token_experts"]) \
        == (4, 16, 7, 4)
    assert c["global_batch"] == 2 * cfg.T and c["parallelism"] == "replicas x2"
    ids, _ = inputs.make_routing(cfg)
    flat = ids.numpy().reshape(-1)
    want = bench.workload_config(cfg, np.bincount(flat, minlength=cfg.E), world=1)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["config"] == want


def test_gemm_sweep_tile_counts():
    """The K sweep's waves come from these tile counts (128 experts x 256 token
    rows, N = 4096): token-major tiles are 128 tokens x 256 weight rows, BFP16
    runs tile 256 as 128-token tiles, weights-on-M tiles cover 128 output
    features (SiLU*up: the gate and up rows of 128 features)."""
    import bench

    E, rpe, N = 128, 256, 4096
    assert bench.sweep_tiles(True, False, 256, E, rpe, N) == 128 * 2 * 16
    assert bench.sweep_tiles(True, False, 64, E, rpe, N) == 128 * 4 * 16
    assert bench.sweep_tiles(False, True, 256, E, rpe, N) == 128 * 2 * 32
    assert bench.sweep_tiles(False, True, 128, E, rpe, N) == 128 * 2 * 32
    assert bench.sweep_tiles(False, False, 256, E, rpe, N) == 128 * 2 * 16
    assert bench.sweep_tiles(False, True, 64, E, rpe, N) == 128 * 4 * 32
    assert set(bench.SWEEP_CFGS) >= {"l2_bfp16_128", "l1_tm_silu"}
