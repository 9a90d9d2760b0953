"""Run the fp64 oracle over many (sequence, KV head) units on all host cores.

TEST INFRASTRUCTURE: imported only by tests and by the CPU-baseline and reference legs
of the benchmark. It adds no arithmetic of its own: every unit is computed by the
oracle's own functions (``gather_sequence*`` over the unit's block table, then
``attend_one_head`` per query row with the causal window of multi-query decode), one
unit per call, in worker processes started with ``spawn`` (safe after a CUDA context
exists in the parent). The only step here is transport: bf16 cache rows travel as
their 16-bit patterns and are widened to float32 (exactly) before the oracle sees them.

A unit is a dict:
  ``kind``    "bf16", "int8", "fp8_e4m3" or "fp8_e5m2"
  ``k``, ``v``  the unit's blocks of one KV head, [n, 1, bs, D]: uint16 bf16 patterns
              (bf16) or uint8 / int8 codes (one-byte caches)
  ``ks``, ``vs``  [n, 1, bs] float32 scales (one-byte caches only)
  ``table``   [n] block table of the unit (indexes into ``k`` / ``v``)
  ``L``       context length; ``q`` [q_len, rows, D] float64 queries of the KV head
  ``scale``, ``bs``   softmax scale and block size
  ``bytes``, ``tokens``   accounting for throughput (not used by the arithmetic)
Result: [q_len, rows, D] float64, new token i seeing positions 0 .. L - q_len + i.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import time

import numpy as np

from . import paged_attention as pa


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - platforms without affinity
        return os.cpu_count() or 1


def _widen_bf16(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def oracle_unit(u):
    """The oracle on one unit (see the module docstring)."""
    kind, bs, L = u["kind"], u["bs"], int(u["L"])
    table = u["table"]
    if kind == "int8":
        K = pa.gather_sequence_int8(u["k"], u["ks"], table, L, 0, bs)
        V = pa.gather_sequence_int8(u["v"], u["vs"], table, L, 0, bs)
    elif kind.startswith("fp8_"):
        K = pa.gather_sequence_fp8(u["k"], u["ks"], table, L, 0, bs, kind[4:])
        V = pa.gather_sequence_fp8(u["v"], u["vs"], table, L, 0, bs, kind[4:])
    else:
        K = pa.gather_sequence(_widen_bf16(u["k"]), table, L, 0, bs)
        V = pa.gather_sequence(_widen_bf16(u["v"]), table, L, 0, bs)
    q = u["q"]
    n, rows, D = q.shape
    out = np.zeros((n, rows, D), dtype=np.float64)
    if L == 0:
        return out
    for i in range(n):
        visible = max(L - n + i + 1, 0)
        for r in range(rows):
            out[i, r], _ = pa.attend_one_head(q[i, r], K[:visible], V[:visible], u["scale"])
    return out


def _pool(processes):
    return mp.get_context("spawn").Pool(processes)


def map_units(units, processes=None, timeout=900.0):
    """Oracle results of every unit, in order, computed on ``processes`` workers
    (default: every host core). A pool that does not finish within ``timeout`` seconds
    (a worker that could not start, for instance) raises instead of waiting forever."""
    n = min(len(units), processes or host_cores())
    if n <= 1:
        return [oracle_unit(u) for u in units]
    with _pool(n) as pool:
        return pool.map_async(oracle_unit, units, chunksize=1).get(timeout)


def _timed_worker(args):
    units, start_at, seconds = args
    while time.time() < start_at:
        time.sleep(0.001)
    end = start_at + seconds
    done_bytes = done_tokens = count = 0
    i = 0
    while time.time() < end:
        u = units[i % len(units)]
        oracle_unit(u)
        done_bytes += u["bytes"]
        done_tokens += u["tokens"]
        count += 1
        i += 1
    return done_bytes, done_tokens, count, time.time() - start_at


class TimedPool:
    """A pool of spawned workers that run the oracle over a fixed sample of units for
    a set wall time, all starting together: the throughput of the host cores."""

    def __init__(self, processes=None):
        self.processes = processes or host_cores()
        self.pool = _pool(self.processes) if self.processes > 1 else None

    def run(self, units, seconds):
        """(bytes, tokens, units computed, elapsed s) over ``seconds`` of wall time,
        the units dealt round-robin to the workers."""
        n = self.processes
        shares = [units[w::n] or units[:1] for w in range(n)]
        start_at = time.time() + (2.0 if self.pool is not None else 0.0)
        tasks = [(s, start_at, seconds) for s in shares]
        res = self.pool.map_async(_timed_worker, tasks, chunksize=1).get(seconds + 300.0) \
            if self.pool is not None else [_timed_worker(tasks[0])]
        b = sum(r[0] for r in res)
        t = sum(r[1] for r in res)
        c = sum(r[2] for r in res)
        el = max(r[3] for r in res)
        return b, t, c, el

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
            self.pool = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
