#!/usr/bin/env python3
"""Benchmark of batched draft verification (+ D-cut) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ragged17|mtp|block|...]
                    [--temperature T]
    python bench.py --workload ragged<k>   (the ragged sweep's pair k = 0..17, B-major;
                                            the default is ragged17: B=128, V=151936, T=0.7)
    python bench.py --workload draft|draft_greedy   (the drafter's step: spec_draft_sample)
    python bench.py --workload confidence           (spec_draft_confidence on the drafter rows)
    python bench.py --workload dcut_cost            (dcut_allocate_cost + verification)
    python bench.py --shards N ...           (vocabulary-sharded verification: the N shards
                                              of a tensor-parallel target, all on this GPU)
    python bench.py --impl reference ...     (the CPU oracle, timed on the host cores)

One step = one pass of the whole verification path over one batch whose
inputs are already in HBM: spec_verify_sample (row statistics + accept test +
first-rejection scan, then the residual / bonus draw), preceded by
dcut_allocate for the D-cut workload.  The timed region replays CUDA graphs
of those C-ABI calls (the calls themselves are what is captured), bracketed
by a barrier and a device synchronise, timed with CUDA events; inputs rotate
through enough independent sets that their total exceeds twice the L2 size.
Rank 0 prints one JSON line.  Under torchrun every rank verifies its own
independent batches (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from draft_verification_02_b300 import workloads as W  # noqa: E402

METRIC = "verified draft positions/sec and achieved HBM GB/s (fraction of peak) at 1 B300"
UNIT = "positions/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
WORKLOADS = {  # name -> (workload, temperature)
    "mtp": (W.MTP, 1.0),
    "block": (W.BLOCK, 0.7),
    "block_greedy": (W.BLOCK, 0.0),
    "dcut": (W.DCUT, 1.0),
    "tiny": (W.TINY, 1.0),
    # the drafter's step of the block workload: draw 16 tokens per request from
    # the padded drafter rows (spec_draft_sample); its own metric
    "draft": (W.BLOCK, 0.7),
    "draft_greedy": (W.BLOCK, 0.0),
    # prefix confidence q(x) of the drafted tokens from the same drafter rows
    "confidence": (W.BLOCK, 0.7),
    "dcut_cost": (W.DCUT, 1.0),
}
# the ragged sweep: B in {4..128} x V in {32000, 128000, 151936}, K_i ~ U{1..16},
# bf16; pair 17 (B=128, V=151936) is the largest single-GPU configuration and
# the default line
for _k in range(len(W.RAGGED_B) * len(W.RAGGED_V)):
    WORKLOADS[f"ragged{_k}"] = (W.ragged(_k), 0.7)
DEFAULT_WORKLOAD = "ragged17"
DRAFT_WORKLOADS = ("draft", "draft_greedy", "confidence")
# the D-cut workload with the cost-unit scheduler (dcut_allocate_cost) in place
# of the token-budget one: requests are admitted while their summed latency
# cost stays within DCUT_MAX_COST units
COST_WORKLOADS = ("dcut_cost",)
DCUT_MAX_COST = 96.0
DRAFT_METRIC = "drafted positions/sec and achieved HBM GB/s (fraction of peak) at 1 B300"
# the sources of each roofline kernel and of its split (verify_params.cuh
# holds the streaming pass's unit planner): a recorded ncu traffic figure
# holds only while these hash the same
KERNEL_SOURCES = {
    "stream_kernel": ["draft_verification_02_b300/csrc/stream_kernel.cuh",
                      "draft_verification_02_b300/csrc/verify_params.cuh",
                      "draft_verification_02_b300/csrc/common.cuh"],
    "draft_sample_kernel": ["draft_verification_02_b300/csrc/finish_kernel.cuh",
                            "draft_verification_02_b300/csrc/verify_params.cuh",
                            "draft_verification_02_b300/csrc/common.cuh"],
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--temperature", type=float, default=None,
                    help="override the workload's temperature (0 = greedy)")
    ap.add_argument("--graph-steps", type=int, default=500,
                    help="verify steps captured per CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU-oracle baseline sample length")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="time budget of the whole reference run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--shards", type=int, default=0,
                    help="vocabulary-sharded verification: the N shards of a tensor-parallel "
                         "target, all on this GPU (0 = unsharded)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (host-side only)
# ---------------------------------------------------------------------------


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device) -> float:
        if self.pg is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float, device) -> float:
        if self.pg is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def rank_seed_offset(rank: int) -> int:
    """Independent input sets per rank (weak scaling)."""
    return 1000 * rank


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel: str = "stream_kernel") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary line
    '<workload> <kernel> <source hash> <bytes>' in profiles/ncu_traffic.txt,
    valid only while the kernel sources still hash the same."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        want = kernel_source_hash(kernel)
        with open(path) as f:
            for line in f:
                p = line.split()
                if len(p) >= 4 and p[0] == workload and p[1] == kernel and p[2] == want:
                    return float(p[3])
    except FileNotFoundError:
        pass
    return None


def read_stream_reference(nbytes: int, device, reps: int = 20) -> float:
    """GB/s of a plain library read of nbytes (torch sum over a bf16 buffer),
    rotating through enough buffers to exceed twice the L2: what a streaming
    read of this size reaches on this GPU, as context for the roofline."""
    n = max(8, nbytes // 2)
    k = max(2, math.ceil(2.2 * l2_bytes(device) / max(nbytes, 1)))
    k = min(k, 64)
    bufs = [torch.ones(n, dtype=torch.bfloat16, device=device) for _ in range(k)]
    out = torch.empty((), dtype=torch.float32, device=device)
    for b in bufs[:3]:
        torch.sum(b, dim=0, dtype=torch.float32, out=out)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record()
    for r in range(reps):
        torch.sum(bufs[r % k], dim=0, dtype=torch.float32, out=out)
    e1.record()
    torch.cuda.synchronize(device)
    sec = e0.elapsed_time(e1) / 1e3 / reps
    del bufs
    return 2 * n / sec / 1e9


def max_depth_per_cost(kmax: int) -> float:
    """max over d = 1..kmax of d / cost(d), cost the cost-unit scheduler's
    latency table {1: 1.0, 2: 1.2, 4: 1.5, 8: 2.0, 16: 3.0} interpolated
    linearly and clamped at its ends."""
    dep, lat = (1, 2, 4, 8, 16), (1.0, 1.2, 1.5, 2.0, 3.0)

    def cost(d):
        if d <= dep[0]:
            return lat[0]
        if d >= dep[-1]:
            return lat[-1]
        for k in range(4):
            if dep[k] <= d <= dep[k + 1]:
                return lat[k] + (d - dep[k]) / (dep[k + 1] - dep[k]) * (lat[k + 1] - lat[k])
    return max(d / cost(d) for d in range(1, max(1, kmax) + 1))


def inputs_sha256(tensors) -> str:
    """SHA-256 over the bytes of the given tensors (host copies), in order:
    a fingerprint of the synthetic inputs a run measured."""
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


def replay_percentiles(events, steps_per_replay):
    """Median, p10 and p90 of the per-step time (ms) over the timed graph
    replays (events recorded between replays, none inside a graph)."""
    ms = sorted(events[q].elapsed_time(events[q + 1]) / steps_per_replay
                for q in range(len(events) - 1))
    if not ms:
        return None

    def pct(x):
        return ms[min(len(ms) - 1, int(round(x * (len(ms) - 1))))]
    return {"replays": len(ms), "steps_per_replay": steps_per_replay, "median": pct(0.5),
            "p10": pct(0.1), "p90": pct(0.9)}


def workload_of(args):
    """(workload, temperature) of the command line."""
    w, T = WORKLOADS[args.workload]
    if args.temperature is not None:
        if args.temperature < 0:
            raise SystemExit("--temperature must be >= 0")
        T = float(args.temperature)
    return w, T


def traffic_key(args, T):
    """The profiles/ncu_traffic.txt key of a bench line: the workload's name,
    with _T<temperature> when --temperature changes the workload's own."""
    T0 = WORKLOADS[args.workload][1]
    return args.workload if T == T0 else f"{args.workload}_T{T:g}"


def workload_desc(w, T, name=None):
    extra = (f", cost-unit D-cut (dcut_allocate_cost, max_cost {DCUT_MAX_COST})"
             if name in COST_WORKLOADS else "")
    return f"{W.describe(w)}, T={T}{extra}"


def l2_bytes(device) -> int:
    try:
        return int(torch.cuda.get_device_properties(device).L2_cache_size)
    except Exception:
        return 126 * 1024 * 1024


def pci_bus_id(device) -> str:
    try:
        p = torch.cuda.get_device_properties(device)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return ""


class ClockSampler:
    """nvidia-smi sampling SM clocks, power and throttle reasons of this GPU
    (read-only) from before the timed region until stop()."""

    def __init__(self, device, enabled=True):
        self.proc = None
        self.path = None
        self.file = None
        if not enabled:
            return
        from draft_verification_02_b300 import clocks
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".txt")
        self.file = os.fdopen(fd, "w")
        try:
            self.proc = subprocess.Popen(clocks.command(pci_bus_id(device), 50),
                                         stdout=self.file, stderr=subprocess.STDOUT)
        except OSError as e:
            self.file.write(f"nvidia-smi unavailable: {e}\n")
            self.file.flush()
            self.proc = None

    def wait_first_sample(self, timeout=5.0):
        t_end = time.time() + timeout
        while self.proc is not None and time.time() < t_end:
            try:
                if os.path.getsize(self.path) > 0:
                    return
            except OSError:
                pass
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.file is not None:
            self.file.close()

    def summary(self, t0, t1):
        if self.path is None:
            return {"samples": 0, "error": "clock sampling disabled"}
        from draft_verification_02_b300 import clocks
        s = clocks.summarize(self.path, t0, t1)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        return s


# ---------------------------------------------------------------------------
# host-side oracle sampling (CPU baseline and reference arm)
# ---------------------------------------------------------------------------


def host_arrays(batch):
    def arr(t):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return {"k": arr(batch.k), "cu": arr(batch.cu_draft), "target": arr(batch.target_logits),
            "draft": arr(batch.draft_logits), "tokens": arr(batch.draft_tokens),
            "u_accept": arr(batch.u_accept), "u_final": arr(batch.u_final),
            "stride": batch.draft_stride, "T": batch.temperature}


def oracle_request(orc, h, i):
    """Run the oracle on request i alone; returns its number of verified positions."""
    K = int(h["k"][i])
    t0 = int(h["cu"][i]) + i
    d0 = i * h["stride"] if h["stride"] else int(h["cu"][i])
    cu = np.array([0, K], np.int32)
    tgt = h["target"][t0:t0 + K + 1]
    if h["T"] == 0:
        r = orc.verify_greedy(tgt, h["tokens"][d0:d0 + K], cu)
    else:
        r = orc.verify_sample(tgt, h["draft"][d0:d0 + K], h["tokens"][d0:d0 + K], cu, h["T"],
                              h["u_accept"][d0:d0 + K], h["u_final"][i:i + 1])
    if r.status != orc.OK:
        raise RuntimeError(f"oracle status {r.status}")
    return K


def oracle_sample_rate(h, seconds, threads, max_requests=None):
    """Positions/s of the oracle over whole requests on `threads` host
    threads (the C oracle releases the GIL), for about `seconds`: rounds of
    the batch's requests, each round handed to the pool at once so that no
    thread waits for another's longer request."""
    import oracle as orc
    orc.load()
    B = len(h["k"])
    done_pos = 0
    done_req = 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        while True:
            n = B if not max_requests else max(1, min(B, max_requests - done_req))
            done_pos += sum(ex.map(lambda r: oracle_request(orc, h, r), range(n)))
            done_req += n
            el = time.perf_counter() - t0
            if el >= seconds or (max_requests and done_req >= max_requests):
                break
    el = time.perf_counter() - t0
    return done_pos / el, done_req, el


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def run_ours(args, dist):
    from draft_verification_02_b300 import specverify as sv
    from draft_verification_02_b300.verifier import Verifier

    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    # the sampler process starts now so that it samples well before the timed region
    sampler = ClockSampler(device, enabled=not args.no_clocks)
    dist.init("nccl")
    w, T = workload_of(args)
    is_cost = args.workload in COST_WORKLOADS
    # host bound on target rows for the cost scheduler: an admitted depth d
    # costs cost(d) units, so the admitted depths sum to at most
    # max_cost * max_d d / cost(d)
    rows = (min(w.B * (w.kmax + 1), int(DCUT_MAX_COST * max_depth_per_cost(w.kmax)) + w.B)
            if is_cost else W.max_target_rows(w))
    is_dcut = bool(w.kmax)
    # ragged depths are drawn once: every rotated set verifies the same depth
    # vector (fresh logits and uniforms), so a step's positions and bytes are
    # fixed and the host passes the exact row count as max_target_rows
    depths0 = None
    if not is_dcut and w.k is None:
        depths0 = W.make_depths(w, "cpu", rank_seed_offset(dist.rank))
        rows = int(depths0.sum().item()) + w.B
    v = Verifier(w.B, rows, w.V, device=device)

    # ---- input sets, resident in HBM
    def make_set(rep):
        s = {}
        if is_dcut:
            prob = W.make_dcut_problem(w, device, rep=rep)
            if is_cost:
                depth_d = torch.empty(w.B, dtype=torch.int32, device=device)
                cu_d = torch.empty(w.B + 1, dtype=torch.int32, device=device)
                sv.check(sv.dcut_allocate_cost(prob.conf, prob.kmax, w.B, w.kmax, DCUT_MAX_COST,
                                               depth_d, cu_d, None, v.workspace), "dcut_cost")
                depth = depth_d.cpu()
            else:
                d = v.dcut(prob.conf, prob.kmax, prob.budget)
                depth = d["depth"].cpu()
            b = W.make_verify_batch(w, T, device, rep=rep, depths=depth, draft_stride=w.kmax)
            if b.target_logits.shape[0] < rows:  # pad to the host bound
                t = torch.zeros((rows, w.V), dtype=b.target_logits.dtype, device=device)
                t[:b.target_logits.shape[0]] = b.target_logits
                b.target_logits = t
            s["prob"] = prob
            s["dcut_out"] = {"depth": torch.empty(w.B, dtype=torch.int32, device=device),
                             "cu": torch.empty(w.B + 1, dtype=torch.int32, device=device),
                             "expected": torch.empty(w.B, dtype=torch.float32, device=device)}
        else:
            b = W.make_verify_batch(w, T, device, rep=rep, depths=depths0)
        s["batch"] = b
        s["out"] = v.outputs(b, rows)
        return s

    first = make_set(rank_seed_offset(dist.rank))
    set_bytes = sum(t.numel() * t.element_size() for t in
                    (first["batch"].target_logits, first["batch"].draft_logits))
    n_sets = max(2, min(64, math.ceil(2.2 * l2_bytes(device) / max(set_bytes, 1))))
    sets = [first] + [make_set(rank_seed_offset(dist.rank) + r) for r in range(1, n_sets)]
    batch0 = first["batch"]
    positions = batch0.n_draft          # verified draft positions per step
    alg_bytes = batch0.algorithmic_bytes()

    def step(s, trace_dcut=None, trace_verify=None):
        b = s["batch"]
        cu = b.cu_draft
        if is_dcut:
            if trace_dcut is not None:
                sv.spec_set_trace(trace_dcut)
            d = s["dcut_out"]
            if is_cost:
                sv.dcut_allocate_cost(s["prob"].conf, s["prob"].kmax, w.B, w.kmax, DCUT_MAX_COST,
                                      d["depth"], d["cu"], None, v.workspace)
            else:
                sv.dcut_allocate(s["prob"].conf, s["prob"].kmax, w.B, w.kmax, s["prob"].budget,
                                 0.0, d["depth"], d["cu"], d["expected"], v.workspace)
            cu = d["cu"]
        if trace_verify is not None:
            sv.spec_set_trace(trace_verify)
        o = s["out"]
        if T == 0:
            st = sv.spec_verify_greedy(b.target_logits, b.draft_tokens, cu, b.B, b.V, rows,
                                       b.draft_stride, o["tokens"], o["accept_len"], v.workspace)
        else:
            st = sv.spec_verify_sample(b.target_logits, b.draft_logits, b.draft_tokens, cu, b.B,
                                       b.V, rows, b.draft_stride, T, b.u_accept, b.u_final,
                                       o["tokens"], o["accept_len"], o["p"], o["q"],
                                       v.workspace)
        if trace_dcut is not None or trace_verify is not None:
            sv.spec_set_trace(None)
        return st

    # ---- warm-up (eager), launch count, correctness of statuses
    n0 = sv.spec_kernel_launch_count()
    for k in range(max(1, args.warmup)):
        sv.check(step(sets[k % n_sets]), "warm-up step")
    torch.cuda.synchronize(device)
    launches_per_step = (sv.spec_kernel_launch_count() - n0) // max(1, args.warmup)
    sv.check(v.device_status(), "device status after warm-up")

    # ---- CUDA graphs of G steps with per-kernel trace events
    K = args.steps
    G = max(1, min(K, args.graph_steps))
    n_verify_ev = 3  # before kernel 1, between the kernels, after kernel 2
    stream = torch.cuda.Stream(device)

    def make_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record()
        return evs

    def capture(n_steps, offset, traced):
        evs = [((make_events(2) if is_dcut else None, make_events(n_verify_ev)) if traced
                else (None, None)) for _ in range(n_steps)]
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n_steps):
                step(sets[(offset + k) % n_sets], evs[k][0], evs[k][1])
        return g, evs

    # the timed graphs carry no trace events: an event between the two
    # verification kernels would turn their programmatic dependency into a
    # full serialisation
    g_main = capture(G, 0, False)[0]
    n_rep, rem = divmod(K, G)
    g_rem = capture(rem, n_rep * G, False)[0] if rem else None
    g_traced, ev_main = capture(G, 0, True)
    # one untimed replay so that the graphs' first-launch cost is not timed
    g_main.replay()
    g_traced.replay()
    torch.cuda.synchronize(device)

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler.wait_first_sample(timeout=60.0)
    dist.barrier()
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    rep_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    with torch.cuda.stream(stream):
        start.record(stream)
        rep_ev[0].record(stream)
        for q in range(n_rep):
            g_main.replay()
            rep_ev[q + 1].record(stream)
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize(device)
    t_wall1 = time.time()
    step_dist = replay_percentiles(rep_ev, G)
    dist.barrier()
    # per-kernel durations: one traced replay of G steps right after
    t0e = torch.cuda.Event(enable_timing=True)
    t1e = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0e.record(stream)
        g_traced.replay()
        t1e.record(stream)
    torch.cuda.synchronize(device)
    sampler.stop()
    elapsed_ms = start.elapsed_time(end)
    elapsed_ms_max = dist.max(elapsed_ms, device)
    traced_ms_per_step = t0e.elapsed_time(t1e) / G
    clocks = sampler.summary(t_wall0, t_wall1)
    st_after = v.device_status()
    if st_after != sv.SPEC_OK:
        raise RuntimeError(f"device status after the timed region: {st_after}")

    stream_us = [ev_main[k][1][0].elapsed_time(ev_main[k][1][1]) * 1e3 for k in range(G)]
    finish_us = [ev_main[k][1][1].elapsed_time(ev_main[k][1][2]) * 1e3 for k in range(G)]
    dcut_us = ([ev_main[k][0][0].elapsed_time(ev_main[k][0][1]) * 1e3 for k in range(G)]
               if is_dcut else [])
    rows_mean = statistics.mean(stream_us)

    total_positions = dist.sum(positions * K, device)
    value = total_positions / (elapsed_ms_max / 1e3)
    ms_per_step = elapsed_ms_max / K
    peak, peak_kind = measured_hbm_peak()
    read_ref = read_stream_reference(alg_bytes, device)
    step_gbs = alg_bytes / (ms_per_step / 1e3) / 1e9
    achieved = alg_bytes / (rows_mean / 1e6) / 1e9

    # acceptance statistics of input set 0's last outputs (the quantities the
    # pages report), by the library's own kernel, outside the timed region
    kmax_stats = w.kmax or w.k or w.k_range[1]
    cu0 = first["dcut_out"]["cu"] if is_dcut else batch0.cu_draft
    st = v.acceptance_stats(first["out"]["accept_len"], cu0, kmax_stats)
    reached = st["reached"][:kmax_stats].cpu().numpy()
    accepted = st["accepted"][:kmax_stats].cpu().numpy()
    acc = {"mean_accepted_len": round(float(st["mean"].item()), 4),
           "per_position_rate": [round(float(a_) / float(r_), 4)
                                 for a_, r_ in zip(accepted, reached) if r_ > 0],
           "per_position_reached": reached.tolist()}

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, v, sets, n_sets, is_dcut, T, rows, w, device, positions, dist)

    # ---- CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        h0 = host_arrays(batch0)
        rate, nreq, el = oracle_sample_rate(h0, args.cpu_seconds, threads)
        rate1, nreq1, el1 = oracle_sample_rate(h0, args.cpu_seconds / 3, 1)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{nreq} whole requests of input set 0 ({workload_desc(w, T)}), "
                         f"one oracle call per request on {threads} host threads, {el:.1f} s",
               "single_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                                 "sample": f"{nreq1} whole requests, {el1:.1f} s"}}

    traffic = recorded_traffic(traffic_key(args, T), "stream_kernel")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_dist": step_dist,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": workload_desc(w, T, args.workload), "B": w.B, "V": w.V,
            "logits_dtype": w.dtype,
            "temperature": T, "verified_positions_per_step": positions,
            "target_rows_per_step": batch0.n_target_rows,
            "l2": f"inputs rotate through {n_sets} independent sets "
                  f"({n_sets * set_bytes / 1e6:.0f} MB > 2x L2 of {l2_bytes(device) / 1e6:.0f} MB)",
            "timing": f"CUDA graphs of {G} steps replayed, CUDA events on the launching stream;"
                      " per-kernel times from a traced replay",
            "parallelism": f"{dist.world} GPU(s), independent batches per GPU",
            "inputs_sha256": inputs_sha256(
                [batch0.target_logits, batch0.draft_logits, batch0.draft_tokens, batch0.cu_draft,
                 batch0.u_accept, batch0.u_final]
                + ([first["prob"].conf, first["prob"].kmax] if is_dcut else [])),
            "torch": torch.__version__,
        },
        "requests_per_s": dist.sum(w.B * K, device) / (elapsed_ms_max / 1e3),
        "hbm_gbs_step": step_gbs,
        "hbm_frac_step": step_gbs / peak,
        "hbm_frac_step_of_nominal_8000": step_gbs / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "kernel": "stream_kernel", "achieved": achieved,
                     "peak": peak, "peak_kind": f"of {peak_kind}", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "library_read_same_bytes_gbs": read_ref,
                     "frac_of_library_read": achieved / read_ref,
                     "launch_us_mean": rows_mean},
        "kernels_us": {"stream_kernel": rows_mean,
                       ("finish_greedy_kernel" if T == 0 else "finish_sample_kernel"):
                           statistics.mean(finish_us),
                       ("dcut_cost_kernel" if is_cost else "dcut_kernel"):
                           statistics.mean(dcut_us) if dcut_us else None,
                       "note": "from one traced replay of the step graph after the timed "
                               "region (events between kernels)",
                       "traced_ms_per_step": traced_ms_per_step},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "acceptance": acc,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def run_sharded(args, dist):
    """A verification workload through the vocabulary-sharded calls: the N
    shards of a tensor-parallel target (contiguous column ranges, each shard's
    logits contiguous as on its own rank), run one after the other on this
    GPU.  The exchanges are stood in for by stacking and an element-wise max
    on the same GPU, so no interconnect is measured.  value = verified
    positions/s of the whole N-shard step on one GPU."""
    from draft_verification_02_b300 import specverify as sv
    from draft_verification_02_b300.sharded import Shard, shard_bounds, shard_columns

    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    sampler = ClockSampler(device, enabled=not args.no_clocks)
    dist.init("nccl")
    w, T = workload_of(args)
    if w.kmax or args.workload in DRAFT_WORKLOADS:
        raise SystemExit("--shards applies to the verification workloads (ragged<k>, mtp, block)")
    N = args.shards
    bounds = shard_bounds(w.V, N)
    depths0 = None
    rows = W.max_target_rows(w)
    if w.k is None:
        depths0 = W.make_depths(w, "cpu", rank_seed_offset(dist.rank))
        rows = int(depths0.sum().item()) + w.B
    shards = [Shard(w.B, rows, bounds, r, device=device) for r in range(N)]

    def make_set(rep, keep_full):
        b = W.make_verify_batch(w, T, device, rep=rep, depths=depths0)
        s = {"batch": b, "targets": shard_columns(b.target_logits, bounds),
             "drafts": shard_columns(b.draft_logits if T > 0 else None, bounds),
             "outs": [sh.outputs() for sh in shards]}
        if not keep_full:  # each shard holds only its own columns
            b.target_logits = b.draft_logits = None
        return s

    first = make_set(rank_seed_offset(dist.rank), True)
    batch0 = first["batch"]
    set_bytes = sum(t.numel() * t.element_size() for t in first["targets"] + first["drafts"]
                    if t is not None)
    n_sets = max(2, min(64, math.ceil(2.2 * l2_bytes(device) / max(set_bytes, 1))))
    sets = [first] + [make_set(rank_seed_offset(dist.rank) + r, False) for r in range(1, n_sets)]
    positions = batch0.n_draft
    alg_bytes = batch0.algorithmic_bytes()

    def step(s, ev=None):
        """ev: per shard, events [before the streaming pass, after it, after
        the row merge, after accept, after mass, after draw]."""
        b = s["batch"]
        recs = []
        for r, sh in enumerate(shards):
            if ev is not None:
                sv.spec_set_trace(ev[r][0:3])
            recs.append(sh.row_stats(s["targets"][r], s["drafts"][r], b.draft_tokens, b.cu_draft,
                                     T))
        rows_all = torch.stack(recs)
        for r, sh in enumerate(shards):
            if ev is not None:
                sv.spec_set_trace(ev[r][3:5])
            sh.accept(rows_all, b.draft_tokens, b.cu_draft, T, b.u_accept, s["outs"][r])
        if T > 0:
            masses = []
            for r, sh in enumerate(shards):
                if ev is not None:
                    sv.spec_set_trace(ev[r][5:7])
                masses.append(sh.final_mass(s["targets"][r], s["drafts"][r]))
            mass_all = torch.stack(masses)
            for r, sh in enumerate(shards):
                if ev is not None:
                    sv.spec_set_trace(ev[r][7:9])
                sh.final_draw(s["targets"][r], s["drafts"][r], mass_all, b.u_final,
                              s["outs"][r]["tokens"])
            top = torch.stack([o["tokens"] for o in s["outs"]]).amax(0)
            for o in s["outs"]:
                o["tokens"].copy_(top)
        if ev is not None:
            sv.spec_set_trace(None)

    n0 = sv.spec_kernel_launch_count()
    for k in range(max(1, args.warmup)):
        step(sets[k % n_sets])
    torch.cuda.synchronize(device)
    launches_per_step = (sv.spec_kernel_launch_count() - n0) // max(1, args.warmup)
    for sh in shards:
        sv.check(sv.spec_get_device_status(sh.workspace), "device status after warm-up")

    K = args.steps
    G = max(1, min(K, args.graph_steps))
    stream = torch.cuda.Stream(device)

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record()
        return evs

    def capture(n_steps, offset, traced):
        evs = [[events(9) for _ in range(N)] if traced else None for _ in range(n_steps)]
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n_steps):
                step(sets[(offset + k) % n_sets], evs[k])
        return g, evs

    g_main = capture(G, 0, False)[0]
    n_rep, rem = divmod(K, G)
    g_rem = capture(rem, n_rep * G, False)[0] if rem else None
    g_traced, ev_main = capture(G, 0, True)
    g_main.replay()
    g_traced.replay()
    torch.cuda.synchronize(device)

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler.wait_first_sample(timeout=60.0)
    dist.barrier()
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    rep_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    with torch.cuda.stream(stream):
        start.record(stream)
        rep_ev[0].record(stream)
        for q in range(n_rep):
            g_main.replay()
            rep_ev[q + 1].record(stream)
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize(device)
    t_wall1 = time.time()
    step_dist = replay_percentiles(rep_ev, G)
    dist.barrier()
    with torch.cuda.stream(stream):
        g_traced.replay()
    torch.cuda.synchronize(device)
    sampler.stop()
    for sh in shards:
        sv.check(sv.spec_get_device_status(sh.workspace), "device status after the timed region")
    elapsed_ms_max = dist.max(start.elapsed_time(end), device)
    clocks = sampler.summary(t_wall0, t_wall1)

    def span(a, b_):  # mean over the traced steps of the summed per-shard spans, us
        return statistics.mean(sum(ev_main[k][r][a].elapsed_time(ev_main[k][r][b_])
                                   for r in range(N)) * 1e3 for k in range(G))
    kern = {"stream_kernel": span(0, 1), "shard_rows_kernel": span(1, 2),
            "shard_accept_kernel": span(3, 4)}
    if T > 0:
        kern["shard_mass_kernel"] = span(5, 6)
        kern["shard_draw_kernel"] = span(7, 8)
    stream_sum = kern["stream_kernel"]
    total_positions = dist.sum(positions * K, device)
    value = total_positions / (elapsed_ms_max / 1e3)
    ms_per_step = elapsed_ms_max / K
    peak, peak_kind = measured_hbm_peak()
    step_gbs = alg_bytes / (ms_per_step / 1e3) / 1e9
    achieved = alg_bytes / (stream_sum / 1e6) / 1e9

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        rate, nreq, el = oracle_sample_rate(host_arrays(batch0), args.cpu_seconds, threads)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{nreq} whole requests of input set 0 ({workload_desc(w, T)}) on the "
                         f"whole vocabulary, one oracle call per request on {threads} host "
                         f"threads, {el:.1f} s"}
    name = f"{traffic_key(args, T)}_tp{N}"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_dist": step_dist,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": f"{workload_desc(w, T, args.workload)}; vocabulary split into {N} "
                        f"contiguous shards (a TP={N} target's layout), all {N} on this GPU, "
                        f"the exchanges stood in for on the same GPU",
            "B": w.B, "V": w.V, "shards": N, "shard_bounds": bounds, "logits_dtype": w.dtype,
            "temperature": T, "verified_positions_per_step": positions,
            "target_rows_per_step": batch0.n_target_rows,
            "l2": f"inputs rotate through {n_sets} independent sets "
                  f"({n_sets * set_bytes / 1e6:.0f} MB > 2x L2 of {l2_bytes(device) / 1e6:.0f} MB)",
            "timing": f"CUDA graphs of {G} steps replayed, CUDA events on the launching stream;"
                      " per-kernel times from a traced replay",
            "parallelism": f"{dist.world} GPU(s), independent batches per GPU",
        },
        "hbm_gbs_step": step_gbs, "hbm_frac_step": step_gbs / peak,
        "roofline": {"bound": "hbm", "kernel": "stream_kernel", "achieved": achieved,
                     "peak": peak, "peak_kind": f"of {peak_kind}", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(name, "stream_kernel"),
                     "algorithmic_bytes_per_launch": alg_bytes / N,
                     "launches": N, "launch_us_mean": stream_sum / N},
        "kernels_us": dict(kern, note=f"summed over the {N} shards, one traced replay; the rest "
                                      "of the step is the stand-in exchanges (torch copies)"),
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "e2e": None,
        "cpu_baseline": cpu,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def run_e2e(args, v, sets, n_sets, is_dcut, T, rows, w, device, positions, dist):
    """Same metric through the public C-ABI calls, with every step's inputs
    copied from pinned host memory and its results read back."""
    from draft_verification_02_b300 import specverify as sv
    steps = max(1, min(args.e2e_steps, args.steps))
    names = ["target_logits", "draft_logits", "draft_tokens", "cu_draft", "u_accept", "u_final"]
    host = []
    for s in sets[:min(n_sets, 3)]:
        b = s["batch"]
        hs = {n: getattr(b, n).cpu().pin_memory() for n in names}
        if is_dcut:
            hs["conf"] = s["prob"].conf.cpu().pin_memory()
            hs["kmax"] = s["prob"].kmax.cpu().pin_memory()
        host.append(hs)
    out_host = torch.empty(rows + w.B, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host[0].values())
    d2h = out_host.numel() * out_host.element_size()
    stream = torch.cuda.current_stream(device)

    def one(k):
        s = sets[k % len(host)]
        hs = host[k % len(host)]
        b = s["batch"]
        for n in names:
            getattr(b, n).copy_(hs[n], non_blocking=True)
        cu = b.cu_draft
        if is_dcut:
            s["prob"].conf.copy_(hs["conf"], non_blocking=True)
            s["prob"].kmax.copy_(hs["kmax"], non_blocking=True)
            d = s["dcut_out"]
            if args.workload in COST_WORKLOADS:
                sv.check(sv.dcut_allocate_cost(s["prob"].conf, s["prob"].kmax, w.B, w.kmax,
                                               DCUT_MAX_COST, d["depth"], d["cu"], None,
                                               v.workspace), "dcut_cost")
            else:
                sv.check(sv.dcut_allocate(s["prob"].conf, s["prob"].kmax, w.B, w.kmax,
                                          s["prob"].budget, 0.0, d["depth"], d["cu"],
                                          d["expected"], v.workspace), "dcut")
            cu = d["cu"]
        o = s["out"]
        if T == 0:
            st = sv.spec_verify_greedy(b.target_logits, b.draft_tokens, cu, b.B, b.V, rows,
                                       b.draft_stride, o["tokens"], o["accept_len"], v.workspace)
        else:
            st = sv.spec_verify_sample(b.target_logits, b.draft_logits, b.draft_tokens, cu, b.B,
                                       b.V, rows, b.draft_stride, T, b.u_accept, b.u_final,
                                       o["tokens"], o["accept_len"], o["p"], o["q"],
                                       v.workspace)
        sv.check(st, "verify")
        out_host[:rows].copy_(o["tokens"][:rows], non_blocking=True)
        out_host[rows:].copy_(o["accept_len"], non_blocking=True)

    for k in range(3):
        one(k)
    torch.cuda.synchronize(device)
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        one(k)
    e1.record(stream)
    torch.cuda.synchronize(device)
    dist.barrier()
    ms = dist.max(e0.elapsed_time(e1), device)
    value = dist.sum(positions * steps, device) / (ms / 1e3)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": ms / steps}


# ---------------------------------------------------------------------------
# the drafter's step: spec_draft_sample over B*Kmax padded drafter rows
# ---------------------------------------------------------------------------


def draft_inputs(w, T, device, rep):
    """Drafter logits [B*K][V] (the block workload's draft rows, every request
    drafting K tokens), kmax and the per-row uniforms u_draft."""
    b = W.make_verify_batch(w, T, device, rep=rep)
    g = torch.Generator().manual_seed(w.seed * 7919 + rep)
    u = torch.rand(w.B * w.k, generator=g, dtype=torch.float32).to(device)
    kmax = torch.full((w.B,), w.k, dtype=torch.int32, device=device)
    return {"draft": b.draft_logits, "kmax": kmax, "u": u}


def oracle_draft_rows(orc, d, u, T, rows, tokens=None):
    """The oracle on the given rows (each row on its own): drawn tokens, or
    with `tokens` the confidence q(x) of those drafted tokens."""
    n = len(rows)
    if tokens is None:
        st, tok, conf = orc.draft_sample(d[rows], np.ones(n, np.int32), 1, T, u[rows])
    else:
        st, conf = orc.draft_confidence(d[rows], tokens[rows], np.ones(n, np.int32), T)
    if st != orc.OK:
        raise RuntimeError(f"oracle status {st}")
    return n


def oracle_draft_rate(d, u, T, seconds, threads, rows_per_call=4, tokens=None):
    import oracle as orc
    orc.load()
    n_rows = d.shape[0]
    done = 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        i = 0
        while True:
            chunks = [[(i + k * rows_per_call + j) % n_rows for j in range(rows_per_call)]
                      for k in range(threads)]
            i += threads * rows_per_call
            done += sum(ex.map(lambda r: oracle_draft_rows(orc, d, u, T, r, tokens), chunks))
            if time.perf_counter() - t0 >= seconds:
                break
    el = time.perf_counter() - t0
    return done / el, done, el


def host_draft(x):
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()


def run_draft(args, dist):
    from draft_verification_02_b300 import specverify as sv
    from draft_verification_02_b300.verifier import Verifier

    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    sampler = ClockSampler(device, enabled=not args.no_clocks)
    dist.init("nccl")
    w, T = workload_of(args)
    Kmax, n_rows = w.k, w.B * w.k
    v = Verifier(w.B, w.B * (Kmax + 1), w.V, device=device)
    e = 4 if w.dtype == "f32" else 2
    alg_bytes = n_rows * w.V * e  # every drafter row read once

    def make_set(rep):
        s = draft_inputs(w, T, device, rep)
        s["tokens"] = torch.empty(n_rows, dtype=torch.int32, device=device)
        s["conf"] = torch.empty(n_rows, dtype=torch.float32, device=device)
        if args.workload == "confidence":  # the drafted tokens whose q(x) is asked
            s["drafted"] = W.make_verify_batch(w, T, device, rep=rep).draft_tokens
        return s

    first = make_set(rank_seed_offset(dist.rank))
    n_sets = max(2, min(64, math.ceil(2.2 * l2_bytes(device) / alg_bytes)))
    sets = [first] + [make_set(rank_seed_offset(dist.rank) + r) for r in range(1, n_sets)]

    is_conf = args.workload == "confidence"

    def step(s, trace=None):
        if trace is not None:
            sv.spec_set_trace(trace)
        if is_conf:  # q(x) of drafted tokens (the drawn ones of set s, fixed inputs here)
            st = sv.spec_draft_confidence(s["draft"], s["drafted"], s["kmax"], w.B, Kmax, w.V, T,
                                          s["conf"], v.workspace)
        else:
            st = sv.spec_draft_sample(s["draft"], s["kmax"], w.B, Kmax, w.V, T,
                                      None if T == 0 else s["u"], s["tokens"], s["conf"],
                                      v.workspace)
        if trace is not None:
            sv.spec_set_trace(None)
        return st

    n0 = sv.spec_kernel_launch_count()
    for k in range(max(1, args.warmup)):
        sv.check(step(sets[k % n_sets]), "warm-up step")
    torch.cuda.synchronize(device)
    launches_per_step = (sv.spec_kernel_launch_count() - n0) // max(1, args.warmup)
    sv.check(v.device_status(), "device status after warm-up")

    K = args.steps
    G = max(1, min(K, args.graph_steps))
    stream = torch.cuda.Stream(device)

    # T > 0: one kernel reads and draws (draft_sample_kernel); T = 0: the
    # streaming pass, then the per-row argmax merge; confidence: the streaming
    # pass, then the per-row q(x)
    if args.workload == "confidence":
        kernels = ["stream_kernel", "confidence_kernel"]
    elif T > 0:
        kernels = ["draft_sample_kernel"]
    else:
        kernels = ["stream_kernel", "draft_greedy_kernel"]

    def capture(n_steps, offset, traced):
        evs = []
        for _ in range(n_steps):
            ev = ([torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)]
                  if traced else None)
            for x in ev or []:
                x.record()
            evs.append(ev)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n_steps):
                step(sets[(offset + k) % n_sets], evs[k])
        return g, evs

    g_main = capture(G, 0, False)[0]
    n_rep, rem = divmod(K, G)
    g_rem = capture(rem, n_rep * G, False)[0] if rem else None
    g_traced, ev_tr = capture(G, 0, True)
    g_main.replay()
    g_traced.replay()
    torch.cuda.synchronize(device)

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler.wait_first_sample(timeout=60.0)
    dist.barrier()
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    rep_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    with torch.cuda.stream(stream):
        start.record(stream)
        rep_ev[0].record(stream)
        for q in range(n_rep):
            g_main.replay()
            rep_ev[q + 1].record(stream)
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize(device)
    t_wall1 = time.time()
    step_dist = replay_percentiles(rep_ev, G)
    dist.barrier()
    with torch.cuda.stream(stream):
        g_traced.replay()
    torch.cuda.synchronize(device)
    sampler.stop()
    elapsed_ms_max = dist.max(start.elapsed_time(end), device)
    clocks = sampler.summary(t_wall0, t_wall1)
    sv.check(v.device_status(), "device status after the timed region")
    kernel_us = {name: statistics.mean(ev_tr[k][q].elapsed_time(ev_tr[k][q + 1]) * 1e3
                                       for k in range(G))
                 for q, name in enumerate(kernels)}
    roof_kernel = kernels[0]  # the kernel that reads the rows
    stream_us = kernel_us[roof_kernel]

    value = dist.sum(n_rows * K, device) / (elapsed_ms_max / 1e3)
    ms_per_step = elapsed_ms_max / K
    peak, peak_kind = measured_hbm_peak()
    achieved = alg_bytes / (stream_us / 1e6) / 1e9
    step_gbs = alg_bytes / (ms_per_step / 1e3) / 1e9

    # end to end: drafter logits and uniforms from pinned host memory, tokens
    # and q(x) read back, through the same public call
    e2e = None
    if not args.no_e2e:
        steps = max(1, min(args.e2e_steps, K))
        in_names = ("draft", "kmax", "drafted") if is_conf else ("draft", "kmax", "u")
        host = [{n: sets[k][n].cpu().pin_memory() for n in in_names}
                for k in range(min(n_sets, 3))]
        out_t = torch.empty(n_rows, dtype=torch.int32).pin_memory()
        out_c = torch.empty(n_rows, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host[0].values())
        d2h = out_t.numel() * 4 + out_c.numel() * 4
        cs = torch.cuda.current_stream(device)

        def one(k):
            s, hs = sets[k % len(host)], host[k % len(host)]
            for n in in_names:
                s[n].copy_(hs[n], non_blocking=True)
            sv.check(step(s), "draft step")
            out_t.copy_(s["tokens"], non_blocking=True)
            out_c.copy_(s["conf"], non_blocking=True)

        for k in range(3):
            one(k)
        torch.cuda.synchronize(device)
        dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        for k in range(steps):
            one(k)
        e1.record(cs)
        torch.cuda.synchronize(device)
        dist.barrier()
        ms = dist.max(e0.elapsed_time(e1), device)
        e2e = {"value": dist.sum(n_rows * steps, device) / (ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
               "ms_per_step": ms / steps}

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        hd, hu = host_draft(first["draft"]), host_draft(first["u"])
        ht = host_draft(first["drafted"]) if is_conf else None
        rate, n, el = oracle_draft_rate(hd, hu, T, args.cpu_seconds, threads, tokens=ht)
        rate1, n1, el1 = oracle_draft_rate(hd, hu, T, args.cpu_seconds / 3, 1, tokens=ht)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} drafter rows of input set 0 ({workload_desc(w, T)}), drawn by "
                         f"the oracle 4 rows per call on {threads} host threads, {el:.1f} s",
               "single_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                                 "sample": f"{n1} drafter rows, {el1:.1f} s"}}

    line = {
        "metric": DRAFT_METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_dist": step_dist,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": (f"{'prefix confidence q(x) of the drafted tokens' if is_conf else 'drafter step'}"
                         f" of {workload_desc(w, T)}: {n_rows} rows, Kmax={Kmax}"),
            "B": w.B, "Kmax": Kmax, "V": w.V, "logits_dtype": w.dtype, "temperature": T,
            "drafted_positions_per_step": n_rows,
            "l2": f"inputs rotate through {n_sets} independent sets "
                  f"({n_sets * alg_bytes / 1e6:.0f} MB > 2x L2 of {l2_bytes(device) / 1e6:.0f} MB)",
            "timing": f"CUDA graphs of {G} steps replayed, CUDA events on the launching stream;"
                      " per-kernel times from a traced replay",
            "parallelism": f"{dist.world} GPU(s), independent batches per GPU",
            "inputs_sha256": inputs_sha256(
                [first["draft"], first["kmax"]]
                + ([first["drafted"]] if is_conf else ([first["u"]] if T > 0 else []))),
            "torch": torch.__version__,
        },
        "hbm_gbs_step": step_gbs,
        "hbm_frac_step": step_gbs / peak,
        "roofline": {"bound": "hbm", "kernel": roof_kernel, "achieved": achieved,
                     "peak": peak, "peak_kind": f"of {peak_kind}", "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(args.workload, roof_kernel),
                     "algorithmic_bytes_per_launch": alg_bytes, "launch_us_mean": stream_us},
        "kernels_us": dict(kernel_us, note="from one traced replay of the step graph after "
                                           "the timed region (events between kernels)"),
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def run_reference_draft(args, dist):
    import oracle as orc
    orc.load()
    w, T = workload_of(args)
    s = draft_inputs(w, T, "cpu", 0)
    d, u = host_draft(s["draft"]), host_draft(s["u"])
    tok = (host_draft(W.make_verify_batch(w, T, "cpu", rep=0).draft_tokens)
           if args.workload == "confidence" else None)
    n_rows = d.shape[0]
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle_draft_rows(orc, d, u, T, [0], tok)
    t_row = max(time.perf_counter() - t0, 1e-5)
    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    n = int(max(threads, min(n_rows, per_step * threads / t_row)))
    ex = ThreadPoolExecutor(threads)

    def one(k):
        rows = [(k * n + j) % n_rows for j in range(n)]
        chunks = [rows[c::threads] for c in range(threads) if rows[c::threads]]
        return sum(ex.map(lambda r: oracle_draft_rows(orc, d, u, T, r, tok), chunks))

    for k in range(args.warmup):
        one(k)
    done = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        done += one(k)
    el = time.perf_counter() - t0
    ex.shutdown()
    value = done / el
    what = ("prefix confidence q(x) of the drafted tokens" if args.workload == "confidence"
            else "drafter step")
    desc = f"{what} of {workload_desc(w, T)}: {n_rows} rows"
    print(json.dumps({
        "impl": "reference", "metric": DRAFT_METRIC, "value": value, "unit": UNIT,
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "B": w.B, "Kmax": w.k, "V": w.V, "logits_dtype": w.dtype,
                   "temperature": T, "sample_per_step": f"{n} of {n_rows} rows"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n} drafter rows per step of {desc}, on {threads} host "
                                   "threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------


def run_reference(args, dist):
    if dist.rank != 0:
        return  # the other ranks exit without work
    if args.workload in DRAFT_WORKLOADS:
        return run_reference_draft(args, dist)
    import oracle as orc
    orc.load()
    w, T = workload_of(args)
    if w.kmax:
        prob = W.make_dcut_problem(w, "cpu")
        if args.workload in COST_WORKLOADS:
            o = orc.dcut_schedule_cost(prob.conf.numpy(), prob.kmax.numpy(), DCUT_MAX_COST)
        else:
            o = orc.dcut_allocate(prob.conf.numpy(), prob.kmax.numpy(), prob.budget)
        batch = W.make_verify_batch(w, T, "cpu", depths=torch.from_numpy(o.depth),
                                    draft_stride=w.kmax)
    else:  # the depth vector our arm verifies on rank 0
        batch = W.make_verify_batch(w, T, "cpu", depths=W.make_depths(w, "cpu", 0)
                                    if w.k is None else None)
    h = host_arrays(batch)
    threads = os.cpu_count() or 1
    # size each step's sample of whole requests to the time budget
    t0 = time.perf_counter()
    oracle_request(orc, h, 0)
    t_req = max(time.perf_counter() - t0, 1e-4)
    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    n_req = int(max(1, min(w.B, per_step * threads / t_req)))
    ex = ThreadPoolExecutor(threads)

    def one(k):
        reqs = [(k * n_req + j) % w.B for j in range(n_req)]
        return sum(ex.map(lambda r: oracle_request(orc, h, r), reqs))

    for k in range(args.warmup):
        one(k)
    pos = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        pos += one(k)
    el = time.perf_counter() - t0
    ex.shutdown()
    value = pos / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w, T, args.workload), "B": w.B, "V": w.V,
                   "logits_dtype": w.dtype, "temperature": T,
                   "sample_per_step": f"{n_req} of {w.B} requests"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n_req} whole requests per step of {workload_desc(w, T)}, "
                                   f"one oracle call per request on {threads} host threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
    elif args.workload in DRAFT_WORKLOADS:
        run_draft(args, dist)
    elif args.shards:
        run_sharded(args, dist)
    else:
        run_ours(args, dist)


if __name__ == "__main__":
    main()
