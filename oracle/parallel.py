"""The oracle on every host core: one spawned worker process per core.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Nothing here computes a probability,
a ratio or a sample.  The module moves logit rows to worker processes and calls oracle
functions there, so that slow float64 runs over whole rounds (the stated round counts of the
five workloads, the CPU baseline of the benchmark) use all the host's cores.

Rows travel as their raw bits (bfloat16 as uint16, float32 as float32).  Each worker widens
its rows to float64 exactly when they arrive (bfloat16 -> float32 by the 16-bit shift, then
float32 -> float64), before any timed call, so a timed run measures the oracle's arithmetic
alone.  Workers are spawned, never forked: a process forked after its parent has used a GPU
can hang.

A task is named "module:function"; the worker imports the module and calls
function(store, **kwargs), where store holds the arrays of the last "load".
"""
from __future__ import annotations

import importlib
import multiprocessing as mp
import os
import time

import numpy as np


def exact_f64(raw: np.ndarray, kind: str) -> np.ndarray:
    """float64 copy of raw logit bits: kind "bf16" (uint16 bit patterns) or "f32" (float32)."""
    if kind == "bf16":
        return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if kind == "f32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    raise ValueError(kind)


def _worker(conn):
    store = {}
    while True:
        msg = conn.recv()
        op = msg[0]
        if op == "stop":
            break
        try:
            if op == "load":
                store = {}
                for name, (arr, kind) in msg[1].items():
                    store[name] = exact_f64(arr, kind) if kind else arr
                conn.send(("ok", None, 0.0))
            elif op == "run":
                mod, fn = msg[1].split(":")
                f = getattr(importlib.import_module(mod), fn)
                t0 = time.perf_counter()
                out = f(store, **msg[2])
                conn.send(("ok", out, time.perf_counter() - t0))
            else:
                conn.send(("error", f"unknown op {op}", 0.0))
        except Exception as e:  # reported to the parent, which raises
            conn.send(("error", f"{type(e).__name__}: {e}", 0.0))


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class OraclePool:
    """A fixed set of spawned workers, each with its own pipe.

    load(parts) gives worker i the arrays parts[i] (a dict name -> (array, kind), kind "bf16",
    "f32" or None for arrays passed as they are); run(task, kwargs) calls the task in every
    loaded worker at once and returns (outputs, wall seconds from the first send to the last
    answer).  Workers beyond len(parts) stay idle for that round.
    """

    def __init__(self, workers: int | None = None):
        self.n = max(1, workers or host_cores())
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for _ in range(self.n):
            parent, child = ctx.Pipe()
            p = ctx.Process(target=_worker, args=(child,), daemon=True)
            p.start()
            child.close()
            self.conns.append(parent)
            self.procs.append(p)
        self.loaded = 0

    def _collect(self, count):
        outs, secs = [], []
        for c in self.conns[:count]:
            status, out, dt = c.recv()
            if status != "ok":
                raise RuntimeError(f"oracle worker failed: {out}")
            outs.append(out)
            secs.append(dt)
        return outs, secs

    def load(self, parts):
        if len(parts) > self.n:
            raise ValueError(f"{len(parts)} parts for {self.n} workers")
        for c, part in zip(self.conns, parts):
            c.send(("load", part))
        self._collect(len(parts))
        self.loaded = len(parts)

    def run(self, task: str, kwargs=None, per_worker=None):
        """Run `task` on every loaded worker; per_worker (a list) overrides kwargs per worker."""
        t0 = time.perf_counter()
        for i, c in enumerate(self.conns[:self.loaded]):
            kw = per_worker[i] if per_worker is not None else (kwargs or {})
            c.send(("run", task, kw))
        outs, _ = self._collect(self.loaded)
        return outs, time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            try:
                c.send(("stop",))
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.kill()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def split_ranges(n: int, parts: int):
    """[lo, hi) ranges of n items over at most `parts` workers, as equal as possible."""
    parts = max(1, min(parts, n))
    edges = np.linspace(0, n, parts + 1).round().astype(int)
    return [(int(edges[i]), int(edges[i + 1])) for i in range(parts)]


def verify_chunk(store, K: int, F: int = 0, C: float = 1.0):
    """oracle.verify on the worker's sequences, one call per sequence (as the single-thread
    baseline calls it).  Their draft tokens come from draft_tokens, run once after the load, so
    a timed run of this task is verification alone."""
    from .verify import verify
    al, ot = [], []
    for b in range(store["target"].shape[0]):
        sl = slice(b, b + 1)
        r = verify(store["target"][sl], store["draft"][sl, :K], store["tokens"][sl], store["u"][sl], store["T"][sl],
                   store["top_p"][sl], F, C)
        al.append(r["accept_len"])
        ot.append(r["out_tokens"])
    return {"accept_len": np.concatenate(al), "out_tokens": np.concatenate(ot)}


def draft_tokens(store, K: int, F: int = 0, C: float = 1.0):
    """Draft tokens of the worker's sequences from the oracle's own draft sampler; kept in the
    store for the verify_chunk runs that follow."""
    from .verify import draft_sample
    toks = []
    for b in range(store["draft"].shape[0]):
        sl = slice(b, b + 1)
        toks.append(draft_sample(store["draft"][sl, :K], store["u_draft"][sl, :K], store["T"][sl], store["top_p"][sl],
                                 F, C)["tokens"])
    store["tokens"] = np.concatenate(toks)
    return None
