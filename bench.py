#!/usr/bin/env python
"""Benchmark of libspecverify on the large-batch verification workload.

One step = one sv_verify call over one round of the B=512, K=5, V=128256 bf16 workload (target
logits for K+1 positions, draft logits for K positions, even sequences greedy), i.e. the whole
verification path: statistics pass, accept tests, residual / bonus draws, float-float tier.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank verifies its own batch (weak
scaling, no data-path collective); timing is the maximum over ranks.  --impl reference times
the float64 oracle on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify rounds/sec (B·(K+1)·V logits) and achieved HBM GB/s vs ~8 TB/s peak"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------------------------------
# host-side helpers (also exercised by the CPU multi-process tests)
# ------------------------------------------------------------------------------------------
def rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank verifies its own synthetic batch (weak scaling)."""
    return base_seed + 1009 * rank


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Units processed by all ranks per second, timed by the slowest rank."""
    return units_per_rank * world * 1000.0 / ms_max


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


STATS_PROFILE = os.path.join(ROOT, "profiles", "k_stats_large_batch_b512.md")


def stats_traffic(batch: int):
    """DRAM bytes per statistics-pass launch from the committed ncu summary of the B=512 workload,
    or None when the workload differs or the kernel's sources changed since the capture."""
    import hashlib
    import re
    if batch != 512 or not os.path.exists(STATS_PROFILE):
        return None
    text = open(STATS_PROFILE).read()
    m_t = re.search(r"^traffic_bytes_per_launch: (\d+)", text, re.M)
    m_h = re.search(r"^kernel_source_sha256: ([0-9a-f]{64})\s+\(([^)]*)\)", text, re.M)
    if not (m_t and m_h):
        return None
    h = hashlib.sha256()
    for name in (x.strip() for x in m_h.group(2).split(",")):
        path = os.path.join(ROOT, "speculative_decoding_verification_gb300", "csrc", name)
        if not os.path.exists(path):
            return None
        h.update(open(path, "rb").read())
    return int(m_t.group(1)) if h.hexdigest() == m_h.group(1) else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.strip().split(", ") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                for name, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


CLOCK_LEAD_S = 0.8   # untimed load before the timed region, so that clock samples cover it
CLOCK_TAIL_S = 0.3


def keep_busy(step, seconds: float):
    """Runs step() (untimed) in batches until `seconds` of wall time have passed."""
    import torch
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            step()
        torch.cuda.synchronize()


def _round_parts(w, r, parts, dev):
    """Round r of workload w as the oracle workers' shares of its sequences: raw bf16 rows,
    uniforms, temperatures (generated on `dev`, copied to the host outside any timing)."""
    import torch
    from oracle.parallel import split_ranges
    from synth import workloads as W
    tgt, drf = W.logits(w, r, device=dev)
    u_draft, u, _ = W.round_uniforms(w, r)
    T = W.temperatures(w)
    tp = W.top_ps(w).astype(np.float64)
    t_raw = tgt.view(torch.int16).cpu().numpy().view(np.uint16)
    d_raw = drf.view(torch.int16).cpu().numpy().view(np.uint16)
    del tgt, drf
    return [{"target": (t_raw[lo:hi], "bf16"), "draft": (d_raw[lo:hi], "bf16"), "u": (u[lo:hi], None),
             "u_draft": (u_draft[lo:hi], None), "T": (T[lo:hi], None), "top_p": (tp[lo:hi], None)}
            for lo, hi in split_ranges(w.B, parts)]


def oracle_round_seconds(w, rounds, workers, dev, repeats=1):
    """Wall seconds of the float64 oracle's verification of whole rounds of workload w on
    `workers` spawned processes (the sequences split evenly, one oracle call per sequence).
    For each round index in `rounds` the rows are loaded into the workers, widened to float64
    and the draft tokens drawn by the oracle's own sampler, all untimed; then verification of
    the whole round is timed `repeats` times.  Returns one time per timed run."""
    from oracle.parallel import OraclePool
    times = []
    with OraclePool(workers) as pool:
        for r in rounds:
            pool.load(_round_parts(w, r, pool.n, dev))
            pool.run("oracle.parallel:draft_tokens", {"K": w.K})
            for _ in range(repeats):
                _, sec = pool.run("oracle.parallel:verify_chunk", {"K": w.K})
                times.append(sec)
    return times


# ------------------------------------------------------------------------------------------
def workload(rank: int, batch: int = 512):
    from synth import workloads as W
    base = W.LARGE_BATCH
    return W.scaled(base, seed=rank_seed(base.seed, rank), B=batch)


def config_block(w):
    rows_read = w.B * (w.K + 1) + (w.B // 2) * w.K
    in_bytes = w.B * (2 * w.K + 1) * w.V * 2
    return {"workload": f"large-batch verify: B={w.B}, K={w.K}, V={w.V}, bf16 target and draft logits, T=1, "
                        "even sequences greedy", "B": w.B, "K": w.K, "V": w.V, "dtype": "bf16",
            "greedy_fraction": 0.5,
            "l2": f"inputs ({in_bytes / 1e9:.2f} GB) exceed L2; no flush between steps",
            "logit_bytes_read_per_round": rows_read * w.V * 2,
            "logit_bytes_nominal_per_round": w.B * (w.K + 1) * w.V * 2 * 2}


def run_reference(args, rank, world):
    """The float64 oracle on all host cores (rank 0 only): every step verifies one whole round of
    the workload (512 sequences, the same round each step, as the library's steps do) on one
    spawned process per core."""
    if rank != 0:
        return None
    import torch
    from oracle.parallel import host_cores
    w = workload(0)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    cores = host_cores()
    times = oracle_round_seconds(w, [0], cores, dev, repeats=args.warmup + args.steps)[args.warmup:]
    sec = statistics.mean(times)
    value = 1.0 / sec
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "rounds/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1000.0, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_block(w),
            "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": cores, "kind": "oracle",
                             "sample": f"whole rounds: all 512 sequences of round 0 per step on {cores} spawned "
                                       "processes, float64 numpy oracle, one call per sequence; widening the rows "
                                       "and drawing the draft tokens untimed"},
            "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def filter_rates(sv, dev, world, n):
    """Rounds/s of sv_verify on the two sampled workloads with filters (B=8, K=5, V=128256 bf16,
    T=0.8): top-p 0.9, and top-k 50 ahead of top-p 0.9.  Their inputs (22.6 MB) fit in L2, so a
    256 MB buffer is written between timed calls and each call is timed alone: replayed from a
    CUDA graph of the call, and (stream_calls) through the Python binding."""
    import torch
    from synth import workloads as W
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for name, base in (("top_p", W.SAMPLED_TOPP), ("top_k_top_p", W.SAMPLED_TOPK)):
        w = W.scaled(base, seed=rank_seed(base.seed, int(os.environ.get("RANK", "0"))))
        tgt, drf = W.logits(w, 0, device=dev)
        u_draft, u, _ = W.round_uniforms(w, 0)
        T_d = torch.as_tensor(W.temperatures(w), device=dev)
        tp_d = torch.as_tensor(W.top_ps(w), device=dev)
        tk_d = torch.as_tensor(W.top_ks(w), device=dev) if w.top_k else None
        u_d = torch.as_tensor(u, device=dev)
        toks, _, st = sv.sv_saguaro_sample(drf, torch.as_tensor(u_draft[:, :w.K].copy(), device=dev), T_d, top_p=tp_d,
                                           n_rows=w.K, top_k=tk_d)
        ws = sv.Workspace()
        stats = sv.new_stats(dev)

        def call():
            sv.sv_verify(tgt, drf, toks, u_d, T_d, top_p=tp_d, top_k=tk_d, stats=stats, workspace=ws)
        for _ in range(5):
            call()
        torch.cuda.synchronize()

        def timed(fn):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            barrier(world)
            for b, e in ev:
                flush.fill_(1)
                b.record()
                fn()
                e.record()
            torch.cuda.synchronize()
            return max_over_ranks(statistics.mean(b.elapsed_time(e) for b, e in ev), world)
        ms_stream = timed(call)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        ms = timed(g.replay)
        st = sv.read_stats(stats)
        if st["status"] != 0:
            raise RuntimeError(f"filtered verify failed: {st}")
        out[name] = {"workload": w.name, "value": whole_job_rate(1.0, world, ms), "unit": "rounds/s",
                     "ms_per_round": ms, "timing": "CUDA graph of one call, replayed", "steps": n,
                     "logit_bytes_per_round": round_logit_bytes(w),
                     "l2": "256 MB written between calls",
                     "stream_calls": {"value": whole_job_rate(1.0, world, ms_stream), "unit": "rounds/s",
                                      "ms_per_round": ms_stream},
                     "reresolved": st["reresolved"], "unresolved": st["unresolved"]}
    del flush
    return out


def pyramid_rates(sv, dev, world, n, peak):
    """Rounds/s of one verification stage of three-model speculative decoding (sv_fuzzy_verify):
    qualifier -> target (B=64, K=25, tau 0.5) and draft -> qualifier (B=64, K=12, tau 0.4), the
    fuzzy (divergence) mode, and the assisted mode on the first.  Inputs exceed L2 (0.84 GB and
    0.41 GB): no flush."""
    import torch
    from synth import workloads as W
    out = {}
    cases = (("qualifier_target", W.PYRAMID_QT, "divergence"), ("draft_qualifier", W.PYRAMID_DQ, "divergence"),
             ("qualifier_target_assisted", W.PYRAMID_QT, "assisted"))
    for name, base, mode in cases:
        w = W.scaled(base, seed=rank_seed(base.seed, int(os.environ.get("RANK", "0"))))
        ver, drf = W.logits(w, 0, device=dev)
        u_draft, u, _ = W.round_uniforms(w, 0)
        T_d = torch.as_tensor(W.temperatures(w), device=dev)
        u_d = torch.as_tensor(u, device=dev)
        toks, _, st = sv.sv_saguaro_sample(drf, torch.as_tensor(u_draft[:, :w.K].copy(), device=dev), T_d, n_rows=w.K)
        ws = sv.Workspace()
        stats = sv.new_stats(dev)
        al = torch.empty(w.B, dtype=torch.int32, device=dev)
        ot = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)

        def call():
            sv.sv_fuzzy_verify(ver, drf, toks, u_d, T_d, tau=w.extra["tau"], mode=mode, accept_len=al,
                               out_tokens=ot, stats=stats, workspace=ws)
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        start.record()
        for _ in range(n):
            call()
        end.record()
        torch.cuda.synchronize()
        st = sv.read_stats(stats)
        if st["status"] != 0:
            raise RuntimeError(f"fuzzy verify failed: {st}")
        ms = max_over_ranks(start.elapsed_time(end) / n, world)
        rows = w.B * (2 * w.K + 1)
        byts = rows * w.V * 2
        out[name] = {"workload": w.name, "mode": mode, "value": whole_job_rate(1.0, world, ms), "unit": "rounds/s",
                     "ms_per_round": ms, "steps": n, "rows_per_round": rows, "logit_bytes_per_round": byts,
                     "logit_gbs": byts / (ms * 1e-3) / 1e9, "mean_accept_len": float(al.float().mean().item()),
                     "reresolved": st["reresolved"], "unresolved": st["unresolved"]}
    return out


def mirror_tree(B, kappa, gamma):
    """parents [B, kappa*gamma] of a branch-complete tree: kappa roots below the context, each
    the head of a chain of gamma drafted tokens (node id = branch*gamma + depth, depth 1..gamma)."""
    par = np.zeros((B, kappa * gamma), dtype=np.int64)
    for i in range(kappa):
        for d in range(1, gamma + 1):
            node = i * gamma + d
            par[:, node - 1] = 0 if d == 1 else node - 1
    return par


def tree_rates(sv, dev, world, n):
    """Rounds/s of sv_tree_verify on the branch-complete tree of the Mirror-style workload
    (kappa = 8 roots, depth gamma = 7: 56 drafted nodes, V = 151936 bf16), B = 4 and B = 64
    sequences, T = 1.  Each node's token is the library's draw from its parent's draft row."""
    import torch
    from synth import workloads as W
    out = {}
    for B in (4, 64):
        base = W.MIRROR
        N = base.kappa * base.K
        w = W.scaled(base, B=B, K=N, draft_rows_extra=1, seed=rank_seed(base.seed, int(os.environ.get("RANK", "0"))))
        tgt, drf = W.logits(w, 0, device=dev)
        par = mirror_tree(B, base.kappa, base.K)
        rng = np.random.default_rng(w.seed)
        T_d = torch.as_tensor(W.temperatures(w), device=dev)
        # node tokens: one draw per node from its parent's draft row
        par_d = torch.as_tensor(par, device=dev)
        rows = torch.gather(drf, 1, par_d[:, :, None].expand(B, N, w.V)).contiguous()
        toks, _, _ = sv.sv_saguaro_sample(rows, torch.as_tensor(rng.random((B, N)), device=dev), T_d, n_rows=N)
        u_d = torch.as_tensor(rng.random((B, N + 1)), device=dev)
        par_i = par_d.to(torch.int32)
        ws = sv.Workspace()
        stats = sv.new_stats(dev)
        al = torch.empty(B, dtype=torch.int32, device=dev)
        ot = torch.empty((B, N + 1), dtype=torch.int32, device=dev)

        def call():
            sv.sv_tree_verify(tgt, drf, par_i, toks, u_d, T_d, accept_len=al, out_tokens=ot, path=False, stats=stats,
                              workspace=ws)
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        start.record()
        for _ in range(n):
            call()
        end.record()
        torch.cuda.synchronize()
        st = sv.read_stats(stats)
        if st["status"] != 0:
            raise RuntimeError(f"tree verify failed: {st}")
        ms = max_over_ranks(start.elapsed_time(end) / n, world)
        out[f"mirror_tree_B{B}"] = {"workload": f"branch-complete tree kappa=8 gamma=7 (56 nodes), B={B}, V={w.V} bf16",
                                    "value": whole_job_rate(1.0, world, ms), "unit": "rounds/s", "ms_per_round": ms,
                                    "steps": n, "logit_bytes_per_round": round_logit_bytes(w),
                                    "mean_accept_len": float(al.float().mean().item()),
                                    "child_tests": st["accept_tests"], "reresolved": st["reresolved"],
                                    "unresolved": st["unresolved"],
                                    "l2": "inputs of B=64 exceed L2; B=4 (0.14 GB) fits: no flush"}
    return out


def _timed_calls(call, n, world):
    """Mean ms of n back-to-back calls on the current stream (5 untimed calls first)."""
    import torch
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    start.record()
    for _ in range(n):
        call()
    end.record()
    torch.cuda.synchronize()
    return max_over_ranks(start.elapsed_time(end) / n, world)


def _graph_and_stream(call, n, world):
    """(ms per round replayed from a CUDA graph of one round, ms per round as stream calls).
    The graph holds exactly the library's launches of one round; the stream calls add the
    Python binding's per-call host work."""
    import torch
    ms_stream = _timed_calls(call, n, world)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    return _timed_calls(g.replay, n, world), ms_stream


def whole_call_roofline(bytes_read, ms, peak, peak_kind):
    """The whole verification call as a fraction of the HBM roofline, on the logit bytes it
    actually reads (every target row and the draft rows of sampled sequences for sv_verify; the
    rows up to each first rejection for sv_verify_lazy), over the call's own time."""
    gbs = bytes_read / (ms * 1e-3) / 1e9
    return {"bytes": int(bytes_read), "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
            "peak_source": f"{peak_kind} copy bandwidth", "of_8tbs": gbs / 8000.0}


def round_logit_bytes(w) -> int:
    """Bytes of the logits one round of workload w takes as input: the K+1 target rows and the
    draft rows of every sequence, each read once (the round's HBM floor)."""
    return w.B * (w.K + 1 + w.rows_draft) * w.V * w.elem_bytes


def add_hbm(line, peak):
    """Give each filter, PyramidSD, tree and config line an "hbm" object: its input logit bytes
    per round over its time per round, against the copy bandwidth `peak` (GB/s).  Rounds whose
    inputs sit in L2 and whose time is launch-bound read far below it."""
    for sec in ("filters", "pyramid", "tree", "configs"):
        for v in line.get(sec, {}).values():
            ms = v["ms_per_round"] if "ms_per_round" in v else v["us_per_round"] * 1e-3
            gbs = v["logit_bytes_per_round"] / (ms * 1e-3) / 1e9
            v["hbm"] = {"achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak}


def _round_line(w, n, world, ms_graph, ms_stream, **extra):
    return dict(workload=w.name, value=whole_job_rate(1.0, world, ms_graph), unit="rounds/s",
                us_per_round=ms_graph * 1e3, timing="CUDA graph of one round, replayed", steps=n,
                logit_bytes_per_round=round_logit_bytes(w),
                stream_calls={"value": whole_job_rate(1.0, world, ms_stream), "unit": "rounds/s",
                              "us_per_round": ms_stream * 1e3}, **extra)


def config_rates(sv, dev, world, n):
    """Rounds/s of the other stated workloads, each as the library calls one round makes (inputs
    resident; config 2 is in `filters`), replayed from a CUDA graph of one round (and, beside it,
    as plain stream calls through the Python binding):
      1: B=1, K=4, V=32000 f32 -- one sv_verify call (launch-bound);
      3: SSD / Saguaro, B=16, K=5, V=128256 bf16 -- sv_saguaro_sample (sigma_{8,0.3} draft
         tokens), sv_verify with sigma, sv_cache_keys (fan-out 64), sv_cache_lookup;
      4: Mirror, B=4, kappa=8, gamma=7, V=151936 bf16 -- sv_topk_rows (roots from the early-exit
         row), sv_verify of branch 0 against the early-exit rows, sv_mirror_reuse."""
    import torch
    from synth import workloads as W
    r = int(os.environ.get("RANK", "0"))
    out = {}
    # ---- 1 ----
    w = W.scaled(W.PLAIN, seed=rank_seed(W.PLAIN.seed, r))
    tgt, drf = W.logits(w, 0, device=dev)
    u_draft, u, _ = W.round_uniforms(w, 0)
    T_d = torch.as_tensor(W.temperatures(w), device=dev)
    u_d = torch.as_tensor(u, device=dev)
    toks, _, _ = sv.sv_saguaro_sample(drf, torch.as_tensor(u_draft[:, :w.K].copy(), device=dev), T_d, n_rows=w.K)
    ws, stats = sv.Workspace(), sv.new_stats(dev)
    al = torch.empty(w.B, dtype=torch.int32, device=dev)
    ot = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)

    def call1():
        sv.sv_verify(tgt, drf, toks, u_d, T_d, accept_len=al, out_tokens=ot, stats=stats, workspace=ws)
    out["plain_b1"] = _round_line(w, n, world, *_graph_and_stream(call1, n, world), calls="verify")
    # a graph of 100 consecutive calls, replayed: the per-call device time with no launch gaps
    # between graph replays
    g100 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g100):
        for _ in range(100):
            call1()
    ms100 = _timed_calls(g100.replay, max(1, n // 10), world) / 100
    out["plain_b1"]["graph_of_100_calls"] = {"value": whole_job_rate(1.0, world, ms100), "unit": "rounds/s",
                                             "us_per_round": ms100 * 1e3}
    if sv.read_stats(stats)["status"] != 0:
        raise RuntimeError(f"config 1 failed: {sv.read_stats(stats)}")
    # ---- 3 ----
    w = W.scaled(W.SAGUARO, seed=rank_seed(W.SAGUARO.seed, r))
    tgt, drf = W.logits(w, 0, device=dev)
    u_draft, u, _ = W.round_uniforms(w, 0)
    T_d = torch.as_tensor(W.temperatures(w), device=dev)
    u_d = torch.as_tensor(u, device=dev)
    ud_d = torch.as_tensor(u_draft[:, :w.K].copy(), device=dev)
    _, f_int = sv.sv_fanout(w.budget, w.accept_rate, w.power_r, w.K)
    ws, ws2, ws3, stats = sv.Workspace(), sv.Workspace(), sv.Workspace(), sv.new_stats(dev)
    toks = torch.empty((w.B, w.K), dtype=torch.int32, device=dev)
    al = torch.empty(w.B, dtype=torch.int32, device=dev)
    ot = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)
    keys = torch.empty((w.B, int(sum(f_int))), dtype=torch.int32, device=dev)
    hit = torch.empty(w.B, dtype=torch.uint8, device=dev)

    def call3():
        sv.sv_saguaro_sample(drf, ud_d, T_d, F=w.saguaro_F, C=w.saguaro_C, n_rows=w.K, tokens=toks, workspace=ws2)
        sv.sv_verify(tgt, drf, toks, u_d, T_d, saguaro_F=w.saguaro_F, saguaro_C=w.saguaro_C, accept_len=al,
                     out_tokens=ot, stats=stats, workspace=ws)
        sv.sv_cache_keys(drf, toks, f_int, keys=keys, workspace=ws3)
        sv.sv_cache_lookup(al, ot, keys, f_int, hit=hit)
    out["saguaro_b16"] = _round_line(w, n, world, *_graph_and_stream(call3, n, world),
                                     calls="sample, verify, cache keys, lookup")
    if sv.read_stats(stats)["status"] != 0:
        raise RuntimeError(f"config 3 failed: {sv.read_stats(stats)}")
    # ---- 4 ----
    w = W.scaled(W.MIRROR, seed=rank_seed(W.MIRROR.seed, r))
    tgt, ee = W.logits(w, 0, device=dev)
    _, u, u_branch = W.round_uniforms(w, 0)
    T_d = torch.as_tensor(W.temperatures(w), device=dev)
    u_d = torch.as_tensor(u, device=dev)
    kappa, gamma = w.kappa, w.K
    ee0 = ee[:, 0].contiguous()
    ids, lps, _ = sv.sv_topk_rows(ee0, kappa, T_d)
    branches = torch.zeros((w.B, kappa, gamma), dtype=torch.int32, device=dev)
    branches[:, :, 0] = ids
    for i in range(kappa):   # deeper branch tokens: draws from the early-exit rows (the draft's job)
        ub = torch.as_tensor(u_branch[:, i * gamma + 1:(i + 1) * gamma].copy(), device=dev)
        t_i, _, _ = sv.sv_saguaro_sample(ee[:, 1:].contiguous(), ub, T_d, n_rows=gamma - 1)
        branches[:, i, 1:] = t_i
    toks0 = branches[:, 0, :].contiguous()
    ws, ws2, stats = sv.Workspace(), sv.Workspace(), sv.new_stats(dev)
    al = torch.empty(w.B, dtype=torch.int32, device=dev)
    ot = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)
    reuse = torch.empty(w.B, dtype=torch.uint8, device=dev)

    def call4():
        sv.sv_topk_rows(ee0, kappa, T_d, ids=ids, logprobs=lps, workspace=ws2)
        sv.sv_verify(tgt, ee, toks0, u_d, T_d, accept_len=al, out_tokens=ot, stats=stats, workspace=ws)
        sv.sv_mirror_reuse(branches, al, ot, reuse=reuse)
    out["mirror_b4"] = _round_line(w, n, world, *_graph_and_stream(call4, n, world),
                                   calls="top-kappa roots, verify, reuse")
    if sv.read_stats(stats)["status"] != 0:
        raise RuntimeError(f"config 4 failed: {sv.read_stats(stats)}")
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import speculative_decoding_verification_gb300 as sv
    from speculative_decoding_verification_gb300 import build as _build
    from synth import workloads as W

    _build.build()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    lib = sv.load()
    w = workload(rank, args.batch)
    K, B, V = w.K, w.B, w.V
    tgt, drf = W.logits(w, 0, device=dev)
    u_draft, u, _ = W.round_uniforms(w, 0)
    T = W.temperatures(w)
    T_d = torch.as_tensor(T, device=dev)
    u_d = torch.as_tensor(u, device=dev)
    # draft tokens: the library's own draft sampler (plain p, no transform) at the draft uniforms
    toks_d, _, st = sv.sv_saguaro_sample(drf, torch.as_tensor(u_draft[:, :K].copy(), device=dev), T_d, n_rows=K)
    torch.cuda.synchronize()
    if sv.read_stats(st)["status"] != 0:
        raise RuntimeError(f"draft sampling failed: {sv.read_stats(st)}")
    ws = sv.Workspace()
    al = torch.empty(B, dtype=torch.int32, device=dev)
    ot = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    stats = sv.new_stats(dev)

    lazy = args.path == "lazy"

    def step():
        sv.sv_verify(tgt, drf, toks_d, u_d, T_d, accept_len=al, out_tokens=ot, stats=stats, workspace=ws, lazy=lazy)

    # clocks are sampled over one loaded window around the timed region: nvidia-smi needs a few
    # hundred ms to give its first sample, and K steps take milliseconds, so untimed steps of the
    # same call keep the GPU busy before (after the warm-up) and after the timed region
    clocks = ClockSampler(local_rank)
    clocks.start()
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    keep_busy(step, CLOCK_LEAD_S)
    if sv.read_stats(stats)["status"] != 0:
        raise RuntimeError(f"verify failed: {sv.read_stats(stats)}")

    # ---- timed region: device time of K steps ----
    # The streaming pass's own duration comes from CUDA events the library records around it
    # (the profiling hook), in a second pass of K steps: an event between two kernels stops the
    # next launch from overlapping the previous kernel's tail (programmatic dependent launch),
    # which would add a few microseconds to every step of the headline timing.
    n = args.steps

    def timed(fn):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        for i in range(n):
            fn()
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = start.elapsed_time(end) / n
        st = sv.read_stats(stats)
        if st["status"] != 0:
            raise RuntimeError(f"verify failed: {st}")
        # instrumented pass: the streaming kernel's events, and the step time with them in place
        ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in ev_b + ev_e:
            e.record()          # torch creates the underlying CUDA event on first record
        torch.cuda.synchronize()
        start.record()
        for i in range(n):
            lib.sv_set_profile_events(ev_b[i].cuda_event, ev_e[i].cuda_event)
            fn()
        end.record()
        torch.cuda.synchronize()
        lib.sv_set_profile_events(None, None)
        ms_instr = start.elapsed_time(end) / n
        k_ms = statistics.mean(ev_b[i].elapsed_time(ev_e[i]) for i in range(n))
        st = sv.read_stats(stats)
        if st["status"] != 0:
            raise RuntimeError(f"verify failed: {st}")
        return max_over_ranks(ms, world), k_ms, st, ms_instr

    ms_max, k1_ms, final, ms_instr = timed(step)
    keep_busy(step, CLOCK_TAIL_S)
    clk = clocks.stop()
    clk["window"] = (f"samples every 100 ms from the warm-up to {CLOCK_TAIL_S} s after the timed region; "
                     f"untimed steps keep the GPU busy {CLOCK_LEAD_S} s before and {CLOCK_TAIL_S} s after it")
    value = whole_job_rate(1.0, world, ms_max)

    cfg = config_block(w)
    peak, peak_kind = load_peaks()
    # bytes the streaming pass reads: every needed row (sv_verify), or the rows up to each first
    # rejection (sv_verify_lazy), counted by the library
    k1_bytes = final["rows"] * V * 2
    achieved = k1_bytes / (k1_ms * 1e-3) / 1e9
    line = {"metric": METRIC, "value": value, "unit": "rounds/s", "n_gpus": world, "steps": n, "warmup": args.warmup,
            "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": dict(cfg, path=args.path, bytes_read_per_round=k1_bytes),
            "hbm_gbs_per_step": k1_bytes / (ms_max * 1e-3) / 1e9,
            # the whole call on the logit bytes it reads, against the measured copy bandwidth and
            # the nominal 8 TB/s
            "step_roofline": whole_call_roofline(k1_bytes, ms_max, peak, peak_kind),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": stats_traffic(w.B) if not lazy else None,
                         "kernel": "k_lazy" if lazy else "k_stats",
                         "peak_source": f"{peak_kind} copy bandwidth", "kernel_ms": k1_ms,
                         "timing": "CUDA events around the kernel on its stream, in a second pass of the K steps",
                         "ms_per_step_with_events": ms_instr},
            # per call: k_zero_counters, k_stats, k_accept, k_draw_sums, k_draw_finish, k_exact (eager);
            # k_lazy_init, k_lazy, k_draw_sums, k_draw_finish, k_exact (lazy)
            "gpu_launches": (5 if lazy else 6) * n, "clocks": clk,
            "decisions": {k: final[k] for k in ("accept_tests", "draws", "reresolved", "near_boundary",
                                                "unresolved")}}
    # the other verification path on the same inputs (same outputs; see config.path)
    other = "eager" if lazy else "lazy"
    ms_o, k_o, st_o, _ = timed(lambda: sv.sv_verify(tgt, drf, toks_d, u_d, T_d, accept_len=al, out_tokens=ot,
                                                 stats=stats, workspace=ws, lazy=not lazy))
    b_o = st_o["rows"] * V * 2
    line[other] = {"value": whole_job_rate(1.0, world, ms_o), "unit": "rounds/s", "ms_per_step": ms_o,
                   "bytes_read_per_round": b_o, "kernel": "k_stats" if lazy else "k_lazy", "kernel_ms": k_o,
                   "kernel_gbs": b_o / (k_o * 1e-3) / 1e9, "frac": b_o / (k_o * 1e-3) / 1e9 / peak,
                   "step_roofline": whole_call_roofline(b_o, ms_o, peak, peak_kind)}
    if not args.headline_only:
        line["filters"] = filter_rates(sv, dev, world, min(n, 200))
        line["pyramid"] = pyramid_rates(sv, dev, world, min(n, 200), peak)
        line["tree"] = tree_rates(sv, dev, world, min(n, 200))
        line["configs"] = config_rates(sv, dev, world, min(n, 200))
        add_hbm(line, peak)
    if args.kernel_only:
        return line if rank == 0 else None

    # ---- end to end through the public API with host buffers ----
    tgt_h = tgt.cpu().pin_memory()
    drf_h = drf.cpu().pin_memory()
    tok_h = toks_d.cpu().pin_memory()
    u_h = u_d.cpu().pin_memory()
    T_h = T_d.cpu().pin_memory()
    al_h = torch.empty(B, dtype=torch.int32).pin_memory()
    ot_h = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    d2h = al_h.numel() * 4 + ot_h.numel() * 4
    if not lazy:
        # the library's host entry: it copies the rows the verification reads (every target row,
        # the draft rows of sampled sequences) and the small inputs, verifies, copies back
        ws_h = sv.Workspace()
        moved = []

        def e2e_step():
            _, _, _, m = sv.sv_verify_host(tgt_h, drf_h, tok_h, u_h, T_h, accept_len=al_h, out_tokens=ot_h,
                                           stats=stats, workspace=ws_h)
            moved.append(m)
    else:
        tgt_x = torch.empty_like(tgt)
        drf_x = torch.empty_like(drf)
        tok_x, u_x, T_x = torch.empty_like(toks_d), torch.empty_like(u_d), torch.empty_like(T_d)
        moved = [sum(t.numel() * t.element_size() for t in (tgt_h, drf_h, tok_h, u_h, T_h))]

        def e2e_step():
            for dst, src in ((tgt_x, tgt_h), (drf_x, drf_h), (tok_x, tok_h), (u_x, u_h), (T_x, T_h)):
                dst.copy_(src, non_blocking=True)
            sv.sv_verify(tgt_x, drf_x, tok_x, u_x, T_x, accept_len=al, out_tokens=ot, stats=stats, workspace=ws,
                         lazy=lazy)
            al_h.copy_(al, non_blocking=True)
            ot_h.copy_(ot, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    n2 = max(1, min(n, 10))
    barrier(world)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record()
    for _ in range(n2):
        e2e_step()
    e2.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(s2.elapsed_time(e2) / n2, world)

    h2d = moved[-1]
    line["e2e"] = {"value": whole_job_rate(1.0, world, e2e_ms), "unit": "rounds/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                   "call": "sv_verify_lazy after host copies" if lazy else "sv_verify_host (host buffers)"}
    # ---- CPU baseline: the float64 oracle on whole rounds, all host cores and one (rank 0) ----
    if rank == 0 and world == 1:
        from oracle.parallel import host_cores
        cores = host_cores()
        many = oracle_round_seconds(w, [0, 1, 2, 3, 4], cores, dev)
        one = oracle_round_seconds(w, [0, 1, 2], 1, dev)
        line["cpu_baseline"] = {"value": len(many) / sum(many), "unit": "rounds/s", "cores": cores, "kind": "oracle",
                                "sample": f"5 whole rounds (rounds 0-4, 512 sequences each, half greedy) on {cores} "
                                          "spawned processes; float64 numpy oracle, one call per sequence; widening "
                                          "the rows and drawing the draft tokens untimed",
                                "seconds_per_round": many,
                                "single_thread": {"value": len(one) / sum(one), "unit": "rounds/s", "cores": 1,
                                                  "sample": "3 whole rounds (rounds 0-2) on one process",
                                                  "seconds_per_round": one}}
    return line if rank == 0 else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=512, help="sequences per round (512: the stated workload)")
    ap.add_argument("--path", choices=["eager", "lazy"], default="eager",
                    help="sv_verify (every candidate row) or sv_verify_lazy (rows up to each first rejection)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="report the device-timed steps only (no end-to-end or CPU-baseline measurement)")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the headline workload (and the other verification path) only: no filter, "
                         "PyramidSD, tree or other-workload lines (for profiling runs)")
    args = ap.parse_args()
    rank, world, local_rank = rank_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)     # rank 0 alone; no process group needed
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
