"""Host logic of bench.py on the CPU: the multi-rank helpers under a real
world-size-2 gloo process group, the torchrun launch of the reference arm
(only rank 0 prints), the gate on the recorded DRAM traffic, and the parsing
of the clock samples."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, w, local = bench.dist_setup(world)
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + 5.0 * r, w)   # rank 1 is the slower one
    bench.barrier(w)
    import torch.distributed as dist
    backend = dist.get_backend()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "max": got, "backend": backend}, f)


def test_rank_helpers_world_size_2_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, x in enumerate(res):
        assert x == {"rank": r, "world": 2, "local": r, "max": 15.0, "backend": "gloo"}


def test_single_process_helpers_need_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup(1) == (0, 1, 0)
    bench.barrier(1)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_mixed"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_recorded_traffic_is_gated_by_the_source_hash(monkeypatch):
    rec = os.path.join(ROOT, "profiles", "ffa_bwd_main_kernel_varlen_causal_1m_dram.txt")
    if not os.path.exists(rec):
        pytest.skip("no DRAM record committed")
    want = None
    for line in open(rec):
        if line.startswith("source_sha256:"):
            want = line.split(":", 1)[1].strip()
    assert want and len(want) == 64
    monkeypatch.setattr(bench, "source_sha256", lambda: want)
    assert bench.recorded_traffic("varlen_causal_1m") > 0
    monkeypatch.setattr(bench, "source_sha256", lambda: "0" * 64)
    assert bench.recorded_traffic("varlen_causal_1m") is None
    assert bench.recorded_traffic("no_such_workload") is None


def test_source_hash_is_stable():
    h = bench.source_sha256()
    assert len(h) == 64 and h == bench.source_sha256()


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_parsing(tmp_path):
    rows = ["0, 2070, 2070, 1390.0, 0x0, Not Active, Not Active, Not Active, Active",
            "0, 1980, 2070, 1385.0, 0x0, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 120.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    cs = bench.ClockSampler(0)
    cs.proc = _FakeProc()
    cs.file = open(tmp_path / "c.csv", "w+")
    cs.file.write("\n".join(rows) + "\n")
    out = cs.stop()
    assert out["sm_mhz"] == 2025.0            # median over the two loaded samples
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 3


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 7])
def test_e2e_pipeline_order(steps):
    order = bench.pipeline_order(steps)
    # every step is copied in, computed and copied out exactly once
    for op in ("h2d", "compute", "d2h"):
        assert sorted(i for o, i in order if o == op) == list(range(steps))
    pos = {x: n for n, x in enumerate(order)}
    for i in range(steps):
        # a step's own copies bracket its compute, and steps compute in order
        assert pos[("h2d", i)] < pos[("compute", i)] < pos[("d2h", i)]
        if i > 0:
            assert pos[("compute", i - 1)] < pos[("compute", i)]
        # the next step's inputs are on their way before this step computes
        if i + 1 < steps:
            assert pos[("h2d", i + 1)] < pos[("compute", i)]
        # two buffer sets: a set is refilled only after the step two back has computed on it and
        # copied its results out (the bench waits on those events; their producers come first here)
        if i >= 2:
            assert pos[("compute", i - 2)] < pos[("h2d", i)]
            assert pos[("d2h", i - 2)] < pos[("compute", i)]


def test_secondary_bounds_square_causal():
    """A square causal mask of m 128-row tiles: m(m-1)/2 Full and m Partial blocks in each direction
    (the closed form the planner tests pin).  Executed forward work = 4 d 128^2 per Full block and
    6 d 128^2 per Partial block (the second P.V), per head; backward 10 d 128^2 per block and head."""
    m, hq, d = 8, 4, 128
    L = 128 * m
    info = {"mask_area": L * (L + 1) // 2, "fwd_bm": 128, "fwd_bn": 128, "bwd_bm": 128, "bwd_bn": 128,
            "q2k_full": m * (m - 1) // 2, "q2k_mask": m, "k2q_full": m * (m - 1) // 2, "k2q_mask": m}
    r = bench.secondary_bounds(info, hq, d)
    area_f = 4.0 * info["mask_area"] * hq * d
    fwd_exec = hq * d * 128 * 128 * (4 * m * (m - 1) // 2 + 6 * m)
    bwd_exec = hq * d * 128 * 128 * 10 * (m * (m - 1) // 2 + m)
    assert r["fwd_executed_over_mask_flops"] == pytest.approx(fwd_exec / area_f)
    assert r["bwd_executed_over_mask_flops"] == pytest.approx(bwd_exec / (2.5 * area_f))
    assert r["wasted_mma_frac"]["fwd"] == pytest.approx(1 - area_f / fwd_exec)
    assert r["fwd_exp_per_mask_element"] == pytest.approx(128 * 128 * (m * (m + 1) // 2) / info["mask_area"])
    # a 64-dim head keeps dQ^T at 128 rows: 8 d + 2 * 128 instead of 10 d per block element
    r64 = bench.secondary_bounds(info, hq, 64)
    assert r64["bwd_executed_over_mask_flops"] == pytest.approx(
        hq * 128 * 128 * (8 * 64 + 256) * (m * (m - 1) // 2 + m) / (2.5 * 4.0 * info["mask_area"] * hq * 64))


def test_cta_balance():
    import numpy as np
    # three CTAs starting together at t = 0 ns: busy 10, 20, 30 ms
    tr = np.array([[0, 10_000_000, 3, 30], [0, 20_000_000, 2, 20], [0, 30_000_000, 1, 10]], dtype=np.uint64)
    b = bench.cta_balance(tr)
    assert b["ctas"] == 3 and b["span_ms"] == 30.0
    assert b["busy_max_over_mean"] == pytest.approx(1.5)
    assert b["idle_frac"] == pytest.approx(1 - 60 / 90)
    assert b["units_min_max"] == [1, 3] and b["blocks_max_over_mean"] == pytest.approx(1.5)
    assert bench.cta_balance(np.zeros((0, 4), dtype=np.uint64)) is None


def test_planner_throughput():
    r = bench.planner_throughput({"plan_bytes": 6_000_000, "plan_launches": 40}, 2.0, 6000.0)
    assert r["gbs"] == pytest.approx(3.0) and r["frac_of_hbm"] == pytest.approx(0.0005) and r["launches"] == 40
