#!/usr/bin/env python
"""Benchmark of one paged-KV decode step: append the new token of every request
(paged_kv_append) and attend over the whole paged cache (paged_decode_attention,
split-KV merge included), on seeded synthetic inputs shaped like the pages' workloads.

Prints ONE JSON line (rank 0). ``value`` is achieved HBM throughput in GB/s of
algorithmic bytes (valid KV rows + scales + q + out + used table entries + context
lengths + the appended rows) over the measured step time, summed over ranks; the line
also carries KV tokens/s, the roofline of the decode kernel, an end-to-end figure with
host buffers, clocks, and the CPU oracle timed on a bounded sample.

    python bench.py [--config 7b] [--steps K] [--warmup W] [--gpus N]
    python bench.py --impl reference ...     # the CPU oracle as the reference arm
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_TEXT = {
    "tiny": "tiny: batch 4, 8 q = 8 kv heads, head_dim 64, block 16, context U[1,64], 64-block "
            "permuted pool",
    "7b": "7B-like layer: batch 32, 32 q = 32 kv heads, head_dim 128, context 2048, block 16, "
          "shuffled pool 1.2x demand",
    "70b-gqa": "70B-like GQA: batch 64, 64 q / 8 kv heads, head_dim 128, block 16, context "
               "log-normal (median 1024, sigma 1) clipped [128, 32768]",
    "prefix": "prefix sharing: batch 256, 32 q / 8 kv heads, head_dim 128, block 16, shared "
              "2048-token prefix (128 refcounted blocks) + suffix U[16,512]",
    "int8": "INT8 KV: batch 128, 32 q / 8 kv heads, head_dim 128, context 8192, block 32, "
            "per-token per-head fp32 scales",
    "int8-bs16": "INT8 KV: batch 128, 32 q / 8 kv heads, head_dim 128, context 8192, block 16, "
                 "per-token per-head fp32 scales",
    "fp8-e5m2": "FP8 E5M2 KV: batch 128, 32 q / 8 kv heads, head_dim 128, context 8192, "
                "block 32, per-token per-head fp32 scales",
    "fp8-e4m3": "FP8 E4M3 KV: batch 128, 32 q / 8 kv heads, head_dim 128, context 8192, "
                "block 32, per-token per-head fp32 scales",
    "blocks": "KV block moves on the 7B-like layer's cache (32 kv heads, head_dim 128, block 16, "
              "bf16, 256 KiB per block with V): copy-on-write copy of half the pool, swap-out "
              "of 8 requests (1024 blocks) to pinned host memory and swap-in back",
    "spec-70b": "speculative verification on the 70B-like GQA shape: batch 64, 64 q / 8 kv "
                "heads, head_dim 128, block 16, context log-normal (median 1024, sigma 1) "
                "clipped [128, 32768], q_len 6 new tokens per request (k = 5), causal",
    "spec-70b-q16": "speculative verification on the 70B-like GQA shape with 15 drafted "
                    "tokens: batch 64, 64 q / 8 kv heads, head_dim 128, block 16, context "
                    "log-normal (median 1024, sigma 1) clipped [128, 32768], q_len 16 new "
                    "tokens per request (128 query rows per KV head), causal",
}
L2_BYTES = 129e6
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="7b", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cascade", action="store_true",
                    help="prefix workload: decode through the shared-prefix (cascade) entry point")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# Byte accounting (algorithmic: what the method must move at least once)
# ---------------------------------------------------------------------------

def _one_byte(w):
    """INT8 and FP8 caches: one-byte codes plus one fp32 scale per (token, KV head)."""
    return w.kv_dtype != "bf16"


def decode_bytes(w):
    import numpy as np
    L = w.context_lens.cpu().numpy().astype(np.int64)
    elt = 1 if _one_byte(w) else 2
    tokens = int(L.sum())
    kv = tokens * 2 * w.num_kv_heads * w.head_dim * elt
    scales = tokens * 2 * w.num_kv_heads * 4 if _one_byte(w) else 0
    qo = 2 * w.num_seqs * w.q_len * w.num_q_heads * w.head_dim * 2
    tables = int(sum(-(-int(x) // w.block_size) for x in L)) * 4
    return {"kv": kv, "scales": scales, "q_out": qo, "tables": tables + 4 * w.num_seqs,
            "total": kv + scales + qo + tables + 4 * w.num_seqs, "tokens": tokens}


def append_bytes(w):
    T = int((w.slot_mapping >= 0).sum().item())
    elt = 1 if _one_byte(w) else 2
    rows = T * 2 * w.num_kv_heads * w.head_dim
    scales = T * 2 * w.num_kv_heads * 4 if _one_byte(w) else 0
    return rows * 2 + rows * elt + scales + 8 * w.slot_mapping.numel()


def unique_kv_bytes(w):
    """Bytes of distinct physical KV rows the step touches (prefix blocks counted once)."""
    import numpy as np
    L = w.context_lens.cpu().numpy()
    bt = w.block_tables.cpu().numpy()
    seen = {}
    for s, Ls in enumerate(L):
        n = -(-int(Ls) // w.block_size)
        for j in range(n):
            fill = min(w.block_size, int(Ls) - j * w.block_size)
            seen[int(bt[s, j])] = max(seen.get(int(bt[s, j]), 0), fill)
    elt = 1 if _one_byte(w) else 2
    return sum(seen.values()) * 2 * w.num_kv_heads * w.head_dim * elt


def source_digest():
    """sha256 (16 hex) of the library sources, to match committed ncu figures."""
    import glob
    import hashlib
    files = sorted(glob.glob(os.path.join(ROOT, "paged_kv_decode_02_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "pagedkv.h"))
    h = hashlib.sha256()
    for f in files:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(config):
    """DRAM bytes per decode call from the committed ncu summary, or None when the
    library sources changed since the capture (or the workload was not captured)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        digest, table = None, {}
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 2 and parts[0] == "source_digest":
                    digest = parts[1]
                elif len(parts) == 3 and parts[0] == "traffic":
                    table[parts[1]] = int(parts[2])
        if digest != source_digest():
            return None
        return table.get(config)
    except OSError:
        return None


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# Clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
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
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(", ") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (the reported baseline and the reference arm)
# ---------------------------------------------------------------------------

def _host_units(w, count, seed=0):
    """Copy `count` (sequence, KV head) units of the workload to host arrays."""
    import numpy as np
    import torch
    rng = np.random.default_rng(seed)
    units = []
    g = w.num_q_heads // w.num_kv_heads
    for _ in range(count):
        s = int(rng.integers(w.num_seqs))
        kvh = int(rng.integers(w.num_kv_heads))
        L = int(w.context_lens[s].item())
        n = -(-L // w.block_size)
        blocks = w.block_tables[s, :n].to(torch.int64)
        qs = w.q[s] if w.q_len > 1 else w.q[s][None]        # [q_len, Hq, D]
        unit = {"L": L, "q": qs[:, kvh * g:(kvh + 1) * g].double().cpu().numpy(),
                "table": np.arange(n)}
        if _one_byte(w):
            unit["k"] = w.k_cache[blocks][:, kvh:kvh + 1].cpu().numpy()
            unit["v"] = w.v_cache[blocks][:, kvh:kvh + 1].cpu().numpy()
            unit["ks"] = w.k_scale[blocks][:, kvh:kvh + 1].cpu().numpy()
            unit["vs"] = w.v_scale[blocks][:, kvh:kvh + 1].cpu().numpy()
        else:
            unit["k"] = w.k_cache[blocks][:, kvh:kvh + 1].double().cpu().numpy()
            unit["v"] = w.v_cache[blocks][:, kvh:kvh + 1].double().cpu().numpy()
        units.append(unit)
    return units


def _oracle_unit(w, u):
    import oracle
    if w.kv_dtype == "int8":
        K = oracle.gather_sequence_int8(u["k"], u["ks"], u["table"], u["L"], 0, w.block_size)
        V = oracle.gather_sequence_int8(u["v"], u["vs"], u["table"], u["L"], 0, w.block_size)
    elif w.kv_dtype.startswith("fp8_"):
        f = w.kv_dtype[4:]
        K = oracle.gather_sequence_fp8(u["k"], u["ks"], u["table"], u["L"], 0, w.block_size, f)
        V = oracle.gather_sequence_fp8(u["v"], u["vs"], u["table"], u["L"], 0, w.block_size, f)
    else:
        K = oracle.gather_sequence(u["k"], u["table"], u["L"], 0, w.block_size)
        V = oracle.gather_sequence(u["v"], u["table"], u["L"], 0, w.block_size)
    n = u["q"].shape[0]
    for i in range(n):                       # causal window of new token i
        visible = max(u["L"] - n + i + 1, 0)
        for qh in u["q"][i]:
            oracle.attend_one_head(qh, K[:visible], V[:visible], w.scale)


def _unit_bytes(w, u):
    elt = 1 if _one_byte(w) else 2
    g = w.num_q_heads // w.num_kv_heads
    b = (u["L"] * 2 * w.head_dim * elt + 2 * w.q_len * g * w.head_dim * 2 +
         4 * len(u["table"]))
    if _one_byte(w):
        b += u["L"] * 2 * 4
    return b


def cpu_baseline(w, seconds):
    units = _host_units(w, 64)
    t0 = time.perf_counter()
    done_bytes = done_tokens = n = 0
    while True:
        u = units[n % len(units)]
        _oracle_unit(w, u)
        done_bytes += _unit_bytes(w, u)
        done_tokens += u["L"]
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "kv_tokens_per_s": done_tokens / el,
            "sample": f"{n} (sequence, kv-head) units of the {w.name} workload "
                      f"({done_tokens} KV tokens, {el:.1f} s, fp64 numpy, one thread)"}


# ---------------------------------------------------------------------------
# The GPU step
# ---------------------------------------------------------------------------

def _kv_code(pk, w):
    return {"bf16": pk.pagedkv.KV_BF16, "int8": pk.pagedkv.KV_INT8,
            "fp8_e4m3": pk.pagedkv.KV_FP8_E4M3, "fp8_e5m2": pk.pagedkv.KV_FP8_E5M2}[w.kv_dtype]


def api_append(pk, w, k, v, slots):
    """The append call for the workload's cache dtype."""
    if w.kv_dtype == "int8":
        pk.paged_kv_append_int8(k, v, w.k_cache, w.v_cache, w.k_scale, w.v_scale, slots)
    elif w.kv_dtype.startswith("fp8_"):
        pk.paged_kv_append_fp8(k, v, w.k_cache, w.v_cache, w.k_scale, w.v_scale, slots,
                               fmt=w.kv_dtype[4:])
    else:
        pk.paged_kv_append(k, v, w.k_cache, w.v_cache, slots)


def api_decode(pk, w, q, tables, lens, out, ws, cascade_blocks=0):
    """The decode call for the workload's cache dtype (cascade when asked)."""
    if w.kv_dtype == "int8":
        pk.paged_decode_attention_int8(q, w.k_cache, w.v_cache, w.k_scale, w.v_scale, tables,
                                       lens, w.scale, out=out, workspace=ws)
    elif w.kv_dtype.startswith("fp8_"):
        pk.paged_decode_attention_fp8(q, w.k_cache, w.v_cache, w.k_scale, w.v_scale, tables,
                                      lens, w.scale, fmt=w.kv_dtype[4:], out=out, workspace=ws)
    elif cascade_blocks:
        pk.paged_decode_attention_cascade(q, w.k_cache, w.v_cache, tables, lens, cascade_blocks,
                                          w.scale, out=out, workspace=ws)
    elif w.q_len > 1:
        pk.paged_decode_attention_multi(q, w.k_cache, w.v_cache, tables, lens, w.scale, out=out,
                                        workspace=ws)
    else:
        pk.paged_decode_attention(q, w.k_cache, w.v_cache, tables, lens, w.scale, out=out,
                                  workspace=ws)


def run_ours(args, rank, world):
    import torch

    import paged_kv_decode_02_gb300 as pk
    from paged_kv_decode_02_gb300 import build_lib
    from paged_kv_decode_02_gb300.workloads import make_workload

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(build_lib.LIB):
        build_lib.build()
    if world > 1:
        torch.distributed.barrier()
    pk.load_library()
    w = make_workload(args.config, device=dev)
    cascade_blocks = w.extra.get("prefix_tokens", 0) // w.block_size if args.cascade else 0
    if args.cascade and (_one_byte(w) or cascade_blocks == 0):
        raise SystemExit("--cascade needs a bf16 workload with a shared prefix (prefix)")
    if cascade_blocks:
        need = pk.cascade_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                          w.block_size, w.num_blocks, w.max_blocks_per_seq,
                                          cascade_blocks)
    elif w.q_len > 1:
        need = pk.multi_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                        w.block_size, w.num_blocks, w.max_blocks_per_seq,
                                        w.q_len)
    else:
        need = pk.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                         w.block_size, w.num_blocks, w.max_blocks_per_seq,
                                         _kv_code(pk, w))
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    out = torch.empty_like(w.q)
    stream = torch.cuda.current_stream(dev)

    def append():
        api_append(pk, w, w.new_k, w.new_v, w.slot_mapping)

    def decode():
        api_decode(pk, w, w.q, w.block_tables, w.context_lens, out, ws, cascade_blocks)

    for _ in range(max(args.warmup, 3)):
        append()
        decode()
    torch.cuda.synchronize(dev)

    # The K timed steps are captured once into a CUDA graph (as a serving loop replays
    # its decode step), so the device time is not bounded by Python launch overhead.
    # No events sit between the kernels: append, decode and merge chain with
    # programmatic dependent launch exactly as in a user's stream.
    K = args.steps
    lib = pk.pagedkv.load_library()
    launches0 = lib.pkv_kernel_launch_count()
    step_graph = capture(K, lambda: (append(), decode()), dev)
    step_launches = lib.pkv_kernel_launch_count() - launches0   # kernels in the K steps
    step_graph.replay()                 # upload + warm replay (untimed)
    torch.cuda.synchronize(dev)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index) if (rank == 0 and not args.no_clocks) else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
        time.sleep(0.3)  # let the sampler start before the timed region
    t_start.record(stream)
    step_graph.replay()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    # roofline of the dominant call: K back-to-back decode calls (decode + merge
    # kernels) in a second timed region, CUDA events on the launching stream
    launches0 = lib.pkv_kernel_launch_count()
    dec_graph = capture(K, decode, dev)
    dec_launches = (lib.pkv_kernel_launch_count() - launches0) // K
    dec_graph.replay()
    torch.cuda.synchronize(dev)
    d_start, d_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d_start.record(stream)
    dec_graph.replay()
    d_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop() if clocks else None
    if world > 1:
        torch.distributed.barrier()
    ms_total = t_start.elapsed_time(t_end)
    dec_ms = d_start.elapsed_time(d_end) / K
    dec_how = ("CUDA events around K back-to-back decode calls (decode + merge kernels, "
               "graph replay) after the K timed steps")
    ms_total = job_time_ms(ms_total, world, dev)
    ms_step = ms_total / K

    db = decode_bytes(w)
    step_bytes = db["total"] + append_bytes(w)
    value = job_throughput(step_bytes, ms_step, world)
    tokens_per_s = world * db["tokens"] / (ms_step * 1e-3)
    peak, peak_kind = measured_peak()
    achieved = db["total"] / (dec_ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, pk, dev, append, out, ws, step_bytes, world, cascade_blocks)

    result = {
        "metric": "paged decode attention: achieved HBM GB/s (% of GB300 peak) and KV tokens/s",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype,
        "data": "synthetic (seeded)",
        "kv_tokens_per_s": round(tokens_per_s, 1),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "config": {"workload": WORKLOAD_TEXT[args.config] + (" (cascade decode)" if cascade_blocks
                                                             else ""),
                   "name": args.config + ("+cascade" if cascade_blocks else ""),
                   "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "num_blocks": w.num_blocks,
                   "kv_tokens": db["tokens"], "step_bytes": step_bytes,
                   "unique_kv_bytes": unique_kv_bytes(w) if args.config == "prefix" else None,
                   "l2": f"inputs larger than L2: {db['kv'] / 1e6:.0f} MB of KV per step vs "
                         f"{L2_BYTES / 1e6:.0f} MB L2, no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": measured_traffic(args.config),
                     "traffic_source": "profiles/decode_traffic.txt (ncu dram bytes read+write, "
                                       "every kernel of one decode call)",
                     "kernel": decode_kernels(w, cascade_blocks, dec_launches),
                     "launches_per_call": dec_launches,
                     "bytes_per_launch": db["total"], "avg_launch_ms": round(dec_ms, 5),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs copy bandwidth)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "timing": dec_how},
        "gpu_launches": step_launches,
        "clocks": clk,
    }
    if e2e is not None:
        result["e2e"] = e2e
    return result, w


def decode_kernels(w, cascade_blocks, launches):
    """Names of the kernels one decode call launches (for the roofline record)."""
    if cascade_blocks:
        return "paged_prefix_kernel + paged_decode_kernel + paged_cascade_merge_kernel"
    rows = w.q_len * w.num_q_heads // w.num_kv_heads        # query rows per KV head
    main = "paged_decode_tc_kernel" if (w.q_len > 1 and 48 <= rows <= 128) else \
        "paged_decode_kernel"
    if launches == 1:
        return main + " (split-KV parts folded inside the kernel, one launch per call)"
    return f"{main} + paged_decode_merge_kernel (one decode call)"


def run_blocks(args, rank, world):
    """Block moves: the copy-on-write copy (HBM to HBM, read + write bytes against the
    copy roofline) and eviction to / return from pinned host memory (GPU-driven over
    NVLink-C2C), each timed with CUDA events over K back-to-back calls."""
    import numpy as np
    import torch

    import paged_kv_decode_02_gb300 as pk
    from paged_kv_decode_02_gb300 import build_lib
    from paged_kv_decode_02_gb300.workloads import make_workload

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(build_lib.LIB):
        build_lib.build()
    if world > 1:
        torch.distributed.barrier()
    pk.load_library()
    w = make_workload("7b", device=dev)
    stream = torch.cuda.current_stream(dev)
    blk_bytes = 2 * w.num_kv_heads * w.block_size * w.head_dim * 2       # K + V of a block
    rng = np.random.default_rng(0)
    perm = rng.permutation(w.num_blocks)
    n = w.num_blocks // 2
    src = torch.tensor(perm[:n], dtype=torch.int32, device=dev)
    dst = torch.tensor(perm[n:2 * n], dtype=torch.int32, device=dev)
    L = w.context_lens.cpu().numpy()
    victims = list(range(8))
    ids_np = np.concatenate([w.block_tables[s, :-(-int(L[s]) // w.block_size)].cpu().numpy()
                             for s in victims])
    ids = torch.tensor(ids_np, dtype=torch.int32, device=dev)
    host_k = torch.empty((len(ids_np),) + tuple(w.k_cache.shape[1:]),
                         dtype=torch.bfloat16).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    K = max(1, min(args.steps, 50))

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / K

    clocks = ClockSampler(dev.index) if (rank == 0 and not args.no_clocks) else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    ms_copy = timed(lambda: pk.copy_blocks(w.k_cache, w.v_cache, src, dst))
    ms_out = timed(lambda: pk.swap_out(w.k_cache, w.v_cache, ids, host_k, host_v))
    ms_in = timed(lambda: pk.swap_in(w.k_cache, w.v_cache, ids, host_k, host_v))
    # the two-step alternative: gather on the device, then one bulk copy to the host
    staged = torch.empty((len(ids_np),) + tuple(w.k_cache.shape[1:]), dtype=torch.bfloat16,
                         device=dev)
    ids64 = ids.long()

    def staged_out():
        torch.index_select(w.k_cache, 0, ids64, out=staged)
        host_k.copy_(staged, non_blocking=True)
        torch.index_select(w.v_cache, 0, ids64, out=staged)
        host_v.copy_(staged, non_blocking=True)
    ms_staged = timed(staged_out)
    clk = clocks.stop() if clocks else None
    ms_copy_job = job_time_ms(ms_copy, world, dev)
    copy_bytes = 2 * n * blk_bytes                     # every byte read once and written once
    swap_bytes = len(ids_np) * blk_bytes
    peak, peak_kind = measured_peak()
    copy_gbs = job_throughput(copy_bytes, ms_copy_job, world)
    return {
        "metric": "KV block moves: copy-on-write block copy GB/s (read + write) against the "
                  "HBM copy roofline; swap-out / swap-in GB/s to pinned host memory",
        "value": round(copy_gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_copy_job, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD_TEXT["blocks"], "name": "blocks",
                   "copy_pairs": n, "copy_bytes": copy_bytes, "swap_blocks": len(ids_np),
                   "swap_bytes": swap_bytes,
                   "l2": f"{copy_bytes / 1e6:.0f} MB moved per copy call vs "
                         f"{L2_BYTES / 1e6:.0f} MB L2, no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(copy_bytes / (ms_copy * 1e-3) / 1e9, 2),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(copy_bytes / (ms_copy * 1e-3) / 1e9 / peak, 4),
                     "traffic": None, "kernel": "paged_block_move_kernel (copy)",
                     "bytes_per_launch": copy_bytes, "avg_launch_ms": round(ms_copy, 5),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs copy bandwidth)"},
        "swap": {"swap_out_gbs": round(swap_bytes / (ms_out * 1e-3) / 1e9, 2),
                 "swap_in_gbs": round(swap_bytes / (ms_in * 1e-3) / 1e9, 2),
                 "swap_out_ms": round(ms_out, 4), "swap_in_ms": round(ms_in, 4),
                 "staged_swap_out_gbs": round(swap_bytes / (ms_staged * 1e-3) / 1e9, 2),
                 "staged": "torch index_select into a device buffer + one copy to host, "
                           "for comparison",
                 "bound": "NVLink-C2C between the GPU and Grace memory"},
        "gpu_launches": 3 * K,
        "clocks": clk,
    }


def blocks_cpu_baseline(seconds):
    """The oracle's block copy on host arrays of the same block shape (bounded)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(0)
    cache = rng.integers(-2 ** 15, 2 ** 15, size=(64, 32, 16, 128),
                         dtype=np.int16)                 # 2-byte elements, 128 KiB per block
    src, dst = list(range(0, 32)), list(range(32, 64))
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.copy_blocks(cache, src, dst)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    moved = n * len(src) * cache[0].nbytes * 2
    return {"value": round(moved / el / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} oracle copy_blocks calls of 32 blocks of 128 KiB (K only) on host "
                      f"arrays, {el:.1f} s, numpy, one thread"}


def job_time_ms(ms_local, world, device):
    """Whole-job time of the timed region: the maximum over ranks (replicas finish
    when the slowest does). With one rank, the local time."""
    if world <= 1:
        return float(ms_local)
    import torch
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank, ms_job, world):
    """Units all ranks processed (bytes) over the whole-job time, in GB/s."""
    return world * bytes_per_rank / (ms_job * 1e-3) / 1e9


def capture(K, fn, dev):
    """CUDA graph of K calls of fn() on a side stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(K):
                fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    return g


def run_e2e(args, w, pk, dev, append_dev, out, ws, step_bytes, world, cascade_blocks=0):
    """Same step through the public API from pinned HOST buffers: per step, copy the
    step's inputs host->device (one copy of a packed buffer), append + decode, copy the
    output device->host."""
    import torch
    stream = torch.cuda.current_stream(dev)
    # the step's inputs packed into one pinned host buffer (256-byte aligned regions) and
    # moved by one copy per step into views of one device buffer
    names = ("q", "new_k", "new_v", "slot_mapping", "block_tables", "context_lens")
    srcs = {n: getattr(w, n).contiguous() for n in names}
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += (srcs[n].numel() * srcs[n].element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    dev_in = {}
    for n in names:
        t = srcs[n]
        nb = t.numel() * t.element_size()
        host_buf[offs[n]:offs[n] + nb].view(t.dtype).copy_(t.reshape(-1).cpu())
        dev_in[n] = dev_buf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = total
    d2h = host_out.numel() * host_out.element_size()

    def step():
        dev_buf.copy_(host_buf, non_blocking=True)
        api_append(pk, w, dev_in["new_k"], dev_in["new_v"], dev_in["slot_mapping"])
        api_decode(pk, w, dev_in["q"], dev_in["block_tables"], dev_in["context_lens"], out, ws,
                   cascade_blocks)
        host_out.copy_(out, non_blocking=True)

    ref = out.clone()
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    # the packed inputs are the device-resident step's inputs: the same result
    if not torch.equal(host_out, ref.cpu()):
        raise RuntimeError("end-to-end step disagrees with the device-resident step")
    K = max(1, min(args.steps, 500))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / K
    return {"value": round(world * step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "steps": K,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def run_reference(args, rank):
    """The CPU oracle as the reference arm: each step runs it, as it stands, on a
    bounded sample of the same workload on the host cores."""
    import torch
    from paged_kv_decode_02_gb300.workloads import make_workload
    if rank != 0:
        return None
    if args.config == "blocks":
        base = blocks_cpu_baseline(min(30.0, 2.0 + 0.05 * (args.steps + args.warmup)))
        return {"impl": "reference",
                "metric": "KV block moves: copy-on-write block copy GB/s (read + write) against "
                          "the HBM copy roofline; swap-out / swap-in GB/s to pinned host memory",
                "value": base["value"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
                "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
                "config": {"workload": WORKLOAD_TEXT["blocks"], "name": "blocks"},
                "cpu_baseline": base,
                "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
    w = make_workload(args.config, device="cuda" if torch.cuda.is_available() else "cpu")
    units = _host_units(w, 16, seed=1)
    budget_s = 150.0
    per_step = max(1e-3, budget_s / max(1, args.steps + args.warmup))
    done_bytes = 0
    done_tokens = 0
    for _ in range(args.warmup):
        _oracle_unit(w, units[0])
    t0 = time.perf_counter()
    n = 0
    for _ in range(args.steps):
        ts = time.perf_counter()
        while True:
            u = units[n % len(units)]
            _oracle_unit(w, u)
            done_bytes += _unit_bytes(w, u)
            done_tokens += u["L"]
            n += 1
            if time.perf_counter() - ts >= per_step:
                break
    el = time.perf_counter() - t0
    value = done_bytes / el / 1e9
    sample = (f"{n} (sequence, kv-head) units of the {args.config} workload per run "
              f"({done_tokens} KV tokens), fp64 numpy oracle, one thread")
    return {
        "impl": "reference",
        "metric": "paged decode attention: achieved HBM GB/s (% of GB300 peak) and KV tokens/s",
        "value": round(value, 6), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * el / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "kv_tokens_per_s": round(done_tokens / el, 1),
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    if args.config == "blocks":
        res = run_blocks(args, rank, world)
        if rank == 0 and not args.no_cpu_baseline:
            res["cpu_baseline"] = blocks_cpu_baseline(min(args.cpu_seconds, 10.0))
    else:
        res, w = run_ours(args, rank, world)
        if rank == 0 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
