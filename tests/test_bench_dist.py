"""The bench's multi-rank host logic on CPU: two gloo ranks, each verifying
its own independent batches (weak scaling, no data-path collective).  Only
the timing reductions (barrier, max and sum over ranks) cross ranks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    from draft_verification_02_b300 import workloads as W
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    elapsed = 10.0 + rank  # a rank's own timing
    mx = d.max(elapsed, "cpu")
    total = d.sum(48.0 * (rank + 1), "cpu")
    # each rank draws its own input sets
    b = W.make_verify_batch(W.TINY, 1.0, "cpu", rep=bench.rank_seed_offset(rank))
    q.put((rank, mx, total, b.target_logits[0, :4].tolist()))
    d.barrier()
    d.close()


def test_two_gloo_ranks_reduce_timing_and_draw_independent_inputs():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert all(r[1] == 11.0 for r in res)          # max over ranks
    assert all(r[2] == 48.0 + 96.0 for r in res)   # sum of units over ranks
    assert res[0][3] != res[1][3]                  # independent batches per rank


def test_reference_arm_other_ranks_exit_without_work(capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.rank, d.world = 1, 2
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.run_reference(args, d)
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_line_in_process(capsys):
    import json
    import sys
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    args = bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "2",
                             "--warmup", "1", "--reference-seconds", "2"])
    bench.run_reference(args, d)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["tiny", "mtp"])
def test_reference_arm_prints_one_line(workload):
    """bench.py --impl reference (the CPU oracle, no GPU) prints one JSON line
    with the contract's keys and the oracle as its CPU baseline."""
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", workload, "--steps", "1", "--warmup", "1",
                          "--reference-seconds", "1"],
                         capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_bench_host_helpers():
    """The bench's host-side helpers: the cost table's depth bound, replay
    percentiles and input fingerprints."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    # d / cost(d) peaks at the largest depth: 16 / 3.0 up to Kmax = 16, then d / 3
    assert bench.max_depth_per_cost(1) == 1.0
    assert bench.max_depth_per_cost(16) == 16 / 3.0
    assert bench.max_depth_per_cost(32) == 32 / 3.0
    # d = 4 costs 1.5 (a table point), d = 3 interpolates 1.2 + 0.5 * 0.3 = 1.35
    assert abs(bench.max_depth_per_cost(4) - 4 / 1.5) < 1e-12

    class Ev:
        def __init__(self, t):
            self.t = t

        def elapsed_time(self, other):
            return other.t - self.t
    ev = [Ev(t) for t in (0.0, 10.0, 30.0, 60.0, 100.0)]  # replays of 10, 20, 30, 40 ms
    d = bench.replay_percentiles(ev, 10)
    assert d["replays"] == 4 and d["p10"] == 1.0 and d["p90"] == 4.0 and d["median"] in (2.0, 3.0)
    a = torch.arange(6, dtype=torch.float32)
    b = torch.tensor([1, 2], dtype=torch.int32)
    assert bench.inputs_sha256([a, b]) == bench.inputs_sha256([a.clone(), b.clone()])
    assert bench.inputs_sha256([a, b]) != bench.inputs_sha256([b, a])


def test_default_workload_is_the_largest_ragged_pair():
    """The default line is the ragged sweep's largest single-GPU pair (B=128,
    V=151936, K_i ~ U{1..16}, T=0.7); --temperature overrides T."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args([])
    w, T = bench.workload_of(args)
    assert (w.B, w.V, w.k_range, w.seed, T) == (128, 151936, (1, 16), 27, 0.7)
    w0, T0 = bench.workload_of(bench.parse_args(["--workload", "ragged0", "--temperature", "0"]))
    assert (w0.B, w0.V, T0) == (4, 32000, 0.0)
    assert "ragged_B128_V151936" in bench.workload_desc(w, T)


def test_traffic_key_names_an_overridden_temperature():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--workload", "ragged17", "--temperature", "0"])
    assert bench.traffic_key(args, 0.0) == "ragged17_T0"
    args = bench.parse_args(["--workload", "block"])
    assert bench.traffic_key(args, bench.WORKLOADS["block"][1]) == "block"
