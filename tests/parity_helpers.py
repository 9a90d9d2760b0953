"""Helpers shared by the GPU parity tests: run the CPU oracle on (parts of) a
workload whose tensors live on the GPU. Nothing here touches the CUDA library."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import parallel
from paged_kv_decode_02_gb300.workloads import host_units

# Bound on |GPU - oracle| for bf16 outputs of decode attention (bf16, INT8 and FP8
# caches).
DECODE_ATOL = 1e-2


def to_f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def sequence_blocks(w, s):
    L = int(w.context_lens[s].item())
    n = -(-L // w.block_size)
    return L, w.block_tables[s, :n].to(torch.int64)


def oracle_outputs(w, pairs=None):
    """Oracle outputs [B, Hq, D] (float64; NaN where not computed) for the (s, h)
    pairs given (all when None). Only each sequence's own blocks are copied to the
    host, then re-indexed 0..n-1 for the oracle's gather."""
    B, Hq, D = w.q.shape
    g = w.group
    out = np.full((B, Hq, D), np.nan)
    want = {}
    for (s, h) in (pairs if pairs is not None else [(s, h) for s in range(B) for h in range(Hq)]):
        want.setdefault(s, set()).add(h)
    q = to_f64(w.q)
    for s, heads in want.items():
        L, blocks = sequence_blocks(w, s)
        if L == 0:
            for h in heads:
                out[s, h] = 0.0
            continue
        table = np.arange(len(blocks))
        kvhs = sorted({h // g for h in heads})
        for kvh in kvhs:
            if w.kv_dtype == "int8":
                kc = w.k_cache[blocks][:, kvh:kvh + 1].cpu().numpy()
                vc = w.v_cache[blocks][:, kvh:kvh + 1].cpu().numpy()
                ks = w.k_scale[blocks][:, kvh:kvh + 1].cpu().numpy()
                vs = w.v_scale[blocks][:, kvh:kvh + 1].cpu().numpy()
                K = oracle.gather_sequence_int8(kc, ks, table, L, 0, w.block_size)
                V = oracle.gather_sequence_int8(vc, vs, table, L, 0, w.block_size)
            elif w.kv_dtype.startswith("fp8_"):
                fmt = w.kv_dtype[4:]
                kc = w.k_cache[blocks][:, kvh:kvh + 1].cpu().numpy()
                vc = w.v_cache[blocks][:, kvh:kvh + 1].cpu().numpy()
                ks = w.k_scale[blocks][:, kvh:kvh + 1].cpu().numpy()
                vs = w.v_scale[blocks][:, kvh:kvh + 1].cpu().numpy()
                K = oracle.gather_sequence_fp8(kc, ks, table, L, 0, w.block_size, fmt)
                V = oracle.gather_sequence_fp8(vc, vs, table, L, 0, w.block_size, fmt)
            else:
                kc = to_f64(w.k_cache[blocks][:, kvh:kvh + 1])
                vc = to_f64(w.v_cache[blocks][:, kvh:kvh + 1])
                K = oracle.gather_sequence(kc, table, L, 0, w.block_size)
                V = oracle.gather_sequence(vc, table, L, 0, w.block_size)
            for h in heads:
                if h // g == kvh:
                    out[s, h], _ = oracle.attend_one_head(q[s, h], K, V, w.scale)
    return out


def max_err(gpu_out, ref, pairs=None):
    got = to_f64(gpu_out)
    if pairs is None:
        assert np.all(np.isfinite(got))
        return float(np.max(np.abs(got - ref)))
    errs = [np.max(np.abs(got[s, h] - ref[s, h])) for (s, h) in pairs]
    assert all(np.all(np.isfinite(got[s, h])) for (s, h) in pairs)
    return float(max(errs))


def sample_pairs(w, n, seed=0):
    rng = np.random.default_rng(seed)
    B, Hq = w.num_seqs, w.num_q_heads
    L = w.context_lens.cpu().numpy()
    picks = {(int(np.argmax(L)), 0), (int(np.argmin(L)), Hq - 1), (0, 0), (B - 1, Hq - 1)}
    while len(picks) < n:
        picks.add((int(rng.integers(B)), int(rng.integers(Hq))))
    return sorted(picks)


def oracle_outputs_multi(w, triples=None):
    """Oracle outputs [B, q_len, Hq, D] (NaN where not computed) of multi-query decode
    for the (s, i, h) triples given (all when None): each sequence's own blocks are
    copied to the host and re-indexed; whole sequences go through
    oracle.decode_attention_multi, single triples through the same causal window."""
    B, n, Hq, D = w.q.shape
    g = w.group
    out = np.full((B, n, Hq, D), np.nan)
    q = to_f64(w.q)
    if triples is None:
        for s in range(B):
            L, blocks = sequence_blocks(w, s)
            if L == 0:
                out[s] = 0.0
                continue
            kc, vc = to_f64(w.k_cache[blocks]), to_f64(w.v_cache[blocks])
            out[s] = oracle.decode_attention_multi(q[s:s + 1], kc, vc,
                                                   np.arange(len(blocks))[None, :], [L],
                                                   w.scale, w.block_size)[0]
        return out
    for (s, i, h) in triples:
        L, blocks = sequence_blocks(w, s)
        if L == 0:
            out[s, i, h] = 0.0
            continue
        kvh = h // g
        table = np.arange(len(blocks))
        K = oracle.gather_sequence(to_f64(w.k_cache[blocks][:, kvh:kvh + 1]), table, L, 0,
                                   w.block_size)
        V = oracle.gather_sequence(to_f64(w.v_cache[blocks][:, kvh:kvh + 1]), table, L, 0,
                                   w.block_size)
        visible = L - n + i + 1
        out[s, i, h], _ = oracle.attend_one_head(q[s, i, h], K[:visible], V[:visible], w.scale)
    return out


def oracle_outputs_all(w):
    """The oracle's whole output of a workload, [B, Hq, D] (or [B, q_len, Hq, D] for
    multi-query decode), computed unit by unit -- every (sequence, KV head) -- in a
    process pool over all host cores (oracle.parallel, the oracle's own functions)."""
    B, Hkv, g = w.num_seqs, w.num_kv_heads, w.group
    pairs = [(s, h) for s in range(B) for h in range(Hkv)]
    res = parallel.map_units(host_units(w, pairs))
    out = np.zeros((B, w.q_len, w.num_q_heads, w.head_dim))
    for (s, h), r in zip(pairs, res):
        out[s, :, h * g:(h + 1) * g] = r
    return out if w.q_len > 1 else out[:, 0]


def oracle_outputs_multi_q8(w):
    """Whole output [B, q_len, Hq, D] of multi-query decode over a one-byte cache from
    oracle.decode_attention_multi_quantized, each sequence's own blocks copied to the
    host and re-indexed."""
    B, n, Hq, D = w.q.shape
    fmt = "int8" if w.kv_dtype == "int8" else w.kv_dtype[4:]
    out = np.zeros((B, n, Hq, D))
    q = to_f64(w.q)
    for s in range(B):
        L, blocks = sequence_blocks(w, s)
        if L == 0:
            continue
        kc, vc = w.k_cache[blocks].cpu().numpy(), w.v_cache[blocks].cpu().numpy()
        ks, vs = w.k_scale[blocks].cpu().numpy(), w.v_scale[blocks].cpu().numpy()
        out[s] = oracle.decode_attention_multi_quantized(
            q[s:s + 1], kc, vc, ks, vs, np.arange(len(blocks))[None, :], [L], w.scale, fmt,
            w.block_size)[0]
    return out
