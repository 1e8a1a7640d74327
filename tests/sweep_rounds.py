"""Stated-rounds parity sweep: every round of the five workloads through the library on the GPU
and through the float64 oracle on all host cores, compared output by output.

    python -m tests.sweep_rounds [--configs 1,2,3,4,5] [--rounds N] [--workers W] [--out FILE]

Each workload runs its stated number of rounds (1000 / 200 / 200 / 200 / 50) from its seed,
round r drawing its logits and uniforms from the seeded generators at round index r:
  1  plain verification, B = 1, K = 4, V = 32000 f32;
  2  sampled verification with top-p 0.9, B = 8, K = 5, V = 128256 bf16, T = 0.8;
  3  the Saguaro round: sigma_{8,0.3} draft tokens, verification with p', cache keys of the
     fan-out (budget 64, a = 0.7, r = 1) and the lookup, B = 16;
  4  the Mirror round: top-8 roots of the early-exit row, branches of depth 7, verification
     along branch 0, reuse, B = 4, V = 151936;
  5  the large batch, B = 512, K = 5, V = 128256 bf16, even sequences greedy.
On the GPU side the draft tokens (and the Mirror roots and branches) are the library's own
draws; on the oracle side they are the oracle's own.  Both are compared, and so are accept
lengths, committed tokens, keys, hits and reuse flags: a mismatch anywhere counts.  The GPU's
sv_stats counters give the draws that went to the float-float tier (reresolved), the draws
whose uniform lay within 1e-6 of a boundary (near_boundary) and the decisions left within
2e-11 of one (unresolved).

Sources: SSD notes §2.2 and §4.4-§5.1; SSD abstract page, "Method"; SpS notes §3, §6;
Mirror-SD notes §3.1-§3.2.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle.parallel import OraclePool, host_cores, split_ranges  # noqa: E402
from synth import workloads as W  # noqa: E402

STATED = {1: 1000, 2: 200, 3: 200, 4: 200, 5: 50}
CONFIGS = W.CONFIGS
UNIT_ROWS = 400            # logit rows per oracle unit (about 0.4 GB of float64 at V = 128256)
STAT_KEYS = ("accept_tests", "draws", "reresolved", "near_boundary", "unresolved")


def raw(t: torch.Tensor):
    """Host copy of a logit tensor as (raw bits, kind) for the oracle workers."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16), "bf16"
    return t.cpu().numpy(), "f32"


def _stats_add(tally, st):
    import speculative_decoding_verification_gb300 as sv
    s = sv.read_stats(st)
    if s["status"] != 0:
        raise RuntimeError(f"library call failed: {s}")
    for k in STAT_KEYS:
        tally[k] = tally.get(k, 0) + s[k]


def gpu_round(cfg, w, r, dev, ws, tally):
    """One round of workload `cfg` through the library.  Returns (GPU outputs, oracle store)."""
    import speculative_decoding_verification_gb300 as sv
    tgt, drf = W.logits(w, r, device=dev)
    u_draft, u, u_branch = W.round_uniforms(w, r)
    T = W.temperatures(w)
    tp = W.top_ps(w)
    T_d = torch.as_tensor(T, device=dev)
    u_d = torch.as_tensor(u, device=dev)
    tp_d = torch.as_tensor(tp, device=dev) if w.top_p < 1.0 else None
    out = {}
    st_s, st_v = sv.new_stats(dev), sv.new_stats(dev)
    if cfg == 4:
        kappa, gamma = w.kappa, w.K
        ee0 = drf[:, 0].contiguous()
        ids, lps, st_r = sv.sv_topk_rows(ee0, kappa, T_d, workspace=ws)
        branches = torch.zeros((w.B, kappa, gamma), dtype=torch.int32, device=dev)
        branches[:, :, 0] = ids
        ee_deep = drf[:, 1:].contiguous()
        for i in range(kappa):
            ub = torch.as_tensor(u_branch[:, i * gamma + 1:(i + 1) * gamma].copy(), device=dev)
            t_i, _, st_b = sv.sv_saguaro_sample(ee_deep, ub, T_d, n_rows=gamma - 1, workspace=ws)
            branches[:, i, 1:] = t_i
        toks = branches[:, 0, :].contiguous()
        al, ot, _, st_v = sv.sv_verify(tgt, drf, toks, u_d, T_d, stats=st_v, workspace=ws)
        reuse = sv.sv_mirror_reuse(branches, al, ot)
        out.update(roots=ids, root_logprobs=lps, branches=branches, reuse=reuse)
    else:
        ud_d = torch.as_tensor(u_draft[:, :w.K].copy(), device=dev)
        toks, _, st_s = sv.sv_saguaro_sample(drf, ud_d, T_d, top_p=tp_d, F=w.saguaro_F, C=w.saguaro_C, n_rows=w.K,
                                             stats=st_s, workspace=ws)
        al, ot, _, st_v = sv.sv_verify(tgt, drf, toks, u_d, T_d, top_p=tp_d, saguaro_F=w.saguaro_F,
                                       saguaro_C=w.saguaro_C, stats=st_v, workspace=ws)
        out["tokens"] = toks
        if cfg == 3:
            _, f_int = sv.sv_fanout(w.budget, w.accept_rate, w.power_r, w.K)
            keys, _ = sv.sv_cache_keys(drf, toks, f_int, workspace=ws)
            out["keys"] = keys
            out["hit"] = sv.sv_cache_lookup(al, ot, keys, f_int)
    out.update(accept_len=al, out_tokens=ot)
    torch.cuda.synchronize()
    _stats_add(tally, st_v)
    if cfg != 4:
        s = sv.read_stats(st_s)
        if s["status"] != 0:
            raise RuntimeError(f"draft sampling failed: {s}")
        tally["sampler_reresolved"] = tally.get("sampler_reresolved", 0) + s["reresolved"]
        tally["sampler_unresolved"] = tally.get("sampler_unresolved", 0) + s["unresolved"]
    gpu = {k: v.cpu().numpy() for k, v in out.items()}
    store = {"target": raw(tgt), "draft": raw(drf), "u": (u, None), "T": (T, None), "top_p": (tp, None),
             "u_draft": (u_draft, None), "u_branch": (u_branch, None)}
    return gpu, store


def _workspace():
    import speculative_decoding_verification_gb300 as sv
    return sv.Workspace()


def _slice(store, lo, hi):
    return {k: (a[lo:hi], kind) for k, (a, kind) in store.items()}


def _stack(pieces):
    return {k: (np.concatenate([p[k][0] for p in pieces]), pieces[0][k][1]) for k in pieces[0]}


def _task(cfg, w):
    if cfg == 4:
        return "tests.sweep_tasks:mirror_round", {"kappa": w.kappa, "gamma": w.K}
    if cfg == 3:
        from oracle import fanout
        return "tests.sweep_tasks:saguaro_round", {"K": w.K, "F": w.saguaro_F, "C": w.saguaro_C,
                                                   "f_int": list(fanout(w.budget, w.accept_rate, w.power_r, w.K)[1])}
    return "tests.sweep_tasks:verify_round", {"K": w.K, "F": w.saguaro_F, "C": w.saguaro_C}


def _compare(cfg, w, gpu, ora, T, res):
    """Add one unit's comparison to the result counters."""
    n = len(ora["accept_len"])
    res["sequences"] += n
    sampled = T > 0
    k = ora["accept_len"]
    res["accept_tests_oracle"] += int(np.minimum(k[sampled] + 1, w.K).sum())
    res["residual_draws_oracle"] += int(sampled.sum())
    bad_al = gpu["accept_len"] != k
    bad_ot = np.any(gpu["out_tokens"] != ora["out_tokens"], axis=1)
    res["accept_len_mismatches"] += int(bad_al.sum())
    res["token_mismatches"] += int(bad_ot.sum())
    if cfg == 4:
        res["sampler_draws_oracle"] += int(sampled.sum()) * w.kappa * (w.K - 1)
        res["root_mismatches"] += int(np.any(gpu["roots"] != ora["roots"], axis=1).sum())
        res["root_logprob_max_abs_diff"] = max(res["root_logprob_max_abs_diff"],
                                               float(np.max(np.abs(gpu["root_logprobs"] - ora["root_logprobs"]))))
        res["sampler_mismatches"] += int(np.any(gpu["branches"] != ora["branches"], axis=(1, 2)).sum())
        res["reuse_mismatches"] += int((gpu["reuse"] != ora["reuse"]).sum())
    else:
        res["sampler_draws_oracle"] += int(sampled.sum()) * w.K
        res["sampler_mismatches"] += int(np.any(gpu["tokens"] != ora["tokens"], axis=1).sum())
    if cfg == 3:
        res["key_mismatches"] += int(np.any(gpu["keys"] != ora["keys"], axis=1).sum())
        res["hit_mismatches"] += int((gpu["hit"] != ora["hit"]).sum())
        res["hits"] += int(ora["hit"].sum())


MISMATCH_KEYS = ("accept_len_mismatches", "token_mismatches", "sampler_mismatches", "root_mismatches",
                 "reuse_mismatches", "key_mismatches", "hit_mismatches")


def sweep_config(cfg, rounds, pool, dev="cuda", log=None, w=None, round_fn=None):
    """Run `rounds` rounds of workload `cfg` (its stated sizes unless `w` is given); returns the
    result counters.  round_fn stands in for gpu_round (the CPU test of this bookkeeping)."""
    w = CONFIGS[cfg] if w is None else w
    round_fn = gpu_round if round_fn is None else round_fn
    task, kw = _task(cfg, w)
    res = {k: 0 for k in ("sequences", "accept_tests_oracle", "residual_draws_oracle", "sampler_draws_oracle",
                          "hits") + MISMATCH_KEYS}
    res["root_logprob_max_abs_diff"] = 0.0
    res.update(config=cfg, workload=w.name, rounds=rounds, seed=w.seed)
    tally = {}
    ws = _workspace()
    rows_per_seq = (w.K + 1) + w.rows_draft
    t0 = time.perf_counter()
    units, gpus, temps = [], [], []   # pending oracle units and the matching GPU outputs

    def flush():
        if not units:
            return
        pool.load(units)
        outs, _ = pool.run(task, kw)
        for g, o, t in zip(gpus, outs, temps):
            _compare(cfg, w, g, o, t, res)
        units.clear()
        gpus.clear()
        temps.clear()

    seq_cap = max(1, UNIT_ROWS // rows_per_seq)
    pend_g, pend_s = [], []       # rounds stacked into the unit being built
    for r in range(rounds):
        g, s = round_fn(cfg, w, r, dev, ws, tally)
        if w.B > seq_cap:
            for lo, hi in split_ranges(w.B, -(-w.B // seq_cap)):
                units.append(_slice(s, lo, hi))
                gpus.append({k: v[lo:hi] for k, v in g.items()})
                temps.append(s["T"][0][lo:hi])
                if len(units) == pool.n:
                    flush()
        else:
            pend_g.append(g)
            pend_s.append(s)
            if (len(pend_g) + 1) * w.B > seq_cap or r == rounds - 1:
                units.append(_stack(pend_s))
                gpus.append({k: np.concatenate([p[k] for p in pend_g]) for k in pend_g[0]})
                temps.append(units[-1]["T"][0])
                pend_g, pend_s = [], []
                if len(units) == pool.n:
                    flush()
        if log and (r + 1) % max(1, rounds // 5) == 0:
            log(f"config {cfg}: {r + 1}/{rounds} rounds, {time.perf_counter() - t0:.0f} s")
    if pend_g:
        units.append(_stack(pend_s))
        gpus.append({k: np.concatenate([p[k] for p in pend_g]) for k in pend_g[0]})
        temps.append(units[-1]["T"][0])
    flush()
    res["gpu_stats"] = tally
    res["decisions_oracle"] = res["accept_tests_oracle"] + res["residual_draws_oracle"] + res["sampler_draws_oracle"]
    res["mismatches"] = sum(res[k] for k in MISMATCH_KEYS)
    res["seconds"] = time.perf_counter() - t0
    return res


def markdown(results, workers, cmd):
    lines = ["# Parity sweep over the stated rounds of the five workloads", "",
             "Every round of each workload through the library on one GB300 and through the float64 oracle on "
             f"{workers} host cores, compared output by output (draft tokens, roots, branches, accept lengths, "
             "committed tokens, cache keys, hits, reuse flags).", "", "Command (from the repository root, after "
             "`python -c \"import __graft_entry__ as g; g.build()\"`):", "", "```", cmd, "```", "",
             "| workload | rounds | sequences | oracle decisions (accept tests + draws + sampler draws) | mismatches "
             "| float-float tier (GPU draws re-resolved) | near a boundary (GPU count, within 1e-6) | unresolved |",
             "|---|---:|---:|---:|---:|---:|---:|---:|"]
    for r in results:
        g = r["gpu_stats"]
        lines.append(f"| {r['workload']} | {r['rounds']} | {r['sequences']} | {r['decisions_oracle']:,} | "
                     f"{r['mismatches']} | {g.get('reresolved', 0) + g.get('sampler_reresolved', 0)} | "
                     f"{g.get('near_boundary', 0)} | {g.get('unresolved', 0) + g.get('sampler_unresolved', 0)} |")
    lines += ["", "Per-workload counters (JSON):", "", "```"]
    lines += [json.dumps(r, sort_keys=True) for r in results]
    lines += ["```", ""]
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--configs", default="1,2,3,4,5")
    ap.add_argument("--rounds", type=int, default=0, help="rounds per workload (0: the stated count)")
    ap.add_argument("--workers", type=int, default=0)
    ap.add_argument("--out", default="")
    args = ap.parse_args()
    from speculative_decoding_verification_gb300 import build
    build.build()
    cfgs = [int(c) for c in args.configs.split(",")]
    workers = args.workers or host_cores()
    results = []
    with OraclePool(workers) as pool:
        for c in cfgs:
            res = sweep_config(c, args.rounds or STATED[c], pool, log=lambda m: print(m, flush=True))
            print(json.dumps(res), flush=True)
            results.append(res)
    if args.out:
        cmd = "python -m tests.sweep_rounds " + " ".join(sys.argv[1:])
        with open(args.out, "w") as f:
            f.write(markdown(results, workers, cmd))
    bad = sum(r["mismatches"] for r in results)
    sys.exit(1 if bad else 0)


if __name__ == "__main__":
    main()
