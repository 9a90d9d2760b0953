"""Pins for the CPU oracle: each check ties it to something other than itself.

* the pages' worked examples (tests/golden/*.json, each citing its page and section),
* closed forms of softmax attention for inputs where the answer is known exactly,
* brute force in 50-digit arithmetic that walks the physical cache instead of the
  block tables,
* invariants that any correct paged attention must satisfy.

The last group plants plausible mistakes in the oracle (on the CPU) and checks that
the pins catch each one.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import paged_attention as pa
from paged_kv_decode_02_gb300.workloads import BlockAllocator, SequenceBlocks, build_tables

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_exact(x):
    """Round float values to bf16-representable float64 (truncating the fp32 mantissa
    with round-to-nearest-even), as the caches hold bf16."""
    import torch
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _random_case(seed, B=3, Hq=4, Hkv=2, D=4, bs=4, max_len=11, nb=None):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(0, max_len + 1, size=B)
    lengths[0] = max(lengths[0], 1)
    tables, _, NB, _ = build_tables(lengths, bs, rng, num_blocks=nb)
    q = _bf16_exact(rng.standard_normal((B, Hq, D)))
    k = _bf16_exact(rng.standard_normal((NB, Hkv, bs, D)))
    v = _bf16_exact(rng.standard_normal((NB, Hkv, bs, D)))
    return q, k, v, tables, lengths


# ---------------------------------------------------------------------------
# The pages' worked examples
# ---------------------------------------------------------------------------

def test_paging_worked_example_block_counts():
    g = _golden("paging_worked_example.json")
    bs = g["block_size"]
    for req in g["requests"]:
        assert oracle.num_blocks_for(req["tokens"], bs) == req["blocks"]
        # the host allocator builds tables of the same size
        alloc = BlockAllocator(64)
        sb = SequenceBlocks(alloc, bs)
        sb.append_tokens(req["tokens"])
        assert len(sb.blocks) == req["blocks"]
        if "fills" in req:
            fills = [min(bs, req["tokens"] - j * bs) for j in range(req["blocks"])]
            assert fills == req["fills"]


def test_paging_worked_example_gather_reads_only_table_prefix():
    """Request A of the page: 47 tokens in blocks [0x47, 0x12, 0x3a]. The gather must
    visit exactly those blocks (16 + 16 + 15 rows) and never the entries after them."""
    g = _golden("paging_worked_example.json")
    req = g["requests"][0]
    bs = g["block_size"]
    table = np.array(req["example_table"] + [10_000, 10_001], dtype=np.int64)  # poison tail
    NB = max(req["example_table"]) + 1
    cache = np.zeros((NB, 1, bs, 2))
    for b in range(NB):
        for o in range(bs):
            cache[b, 0, o] = (b, o)
    rows = oracle.gather_sequence(cache, table, req["tokens"], 0, bs)
    assert rows.shape == (47, 2)
    visited = [tuple(r) for r in rows]
    expect = [(b, o) for j, b in enumerate(req["example_table"]) for o in range(req["fills"][j])]
    assert visited == expect


def test_waste_bound():
    g = _golden("paging_worked_example.json")
    bs = g["block_size"]
    for L in range(1, 3000):
        waste = oracle.num_blocks_for(L, bs) * bs - L
        assert 0 <= waste <= g["max_wasted_tokens_per_request"]


def test_kv_bytes_7b_example():
    g = _golden("kv_bytes_7b.json")
    e = g["example"]
    b1 = oracle.kv_cache_bytes(**e)
    assert b1 == 1_073_741_824
    assert round(b1 / 1e9, 2) == g["printed_gb_single"]
    b32 = oracle.kv_cache_bytes(**{**e, "batch": 32})
    assert round(b32 / 1e9) == g["printed_gb_batch32"]


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def _single_seq(K_rows, V_rows, bs, perm_seed=None):
    """Lay out one sequence's rows [L, Hkv, D] into a paged cache, optionally with a
    permuted physical placement. Returns (k_cache, v_cache, table)."""
    L, Hkv, D = K_rows.shape
    n = oracle.num_blocks_for(L, bs)
    NB = n + 3
    phys = np.arange(NB)
    if perm_seed is not None:
        phys = np.random.default_rng(perm_seed).permutation(NB)
    k = np.full((NB, Hkv, bs, D), np.nan)
    v = np.full((NB, Hkv, bs, D), np.nan)
    for t in range(L):
        k[phys[t // bs], :, t % bs] = K_rows[t]
        v[phys[t // bs], :, t % bs] = V_rows[t]
    table = np.concatenate([phys[:n], [NB + 5]])
    return k, v, table[None, :]


def test_single_token_returns_its_value_row_exactly():
    rng = np.random.default_rng(1)
    D = 8
    K = rng.standard_normal((1, 1, D))
    V = rng.standard_normal((1, 1, D))
    k, v, tbl = _single_seq(K, V, 16, perm_seed=3)
    q = rng.standard_normal((1, 1, D)) * 100.0
    out = oracle.decode_attention(q, k, v, tbl, [1], scale=0.37)
    assert np.array_equal(out[0, 0], V[0, 0])


def test_zero_scale_gives_mean_of_values():
    rng = np.random.default_rng(2)
    L, D = 37, 8
    K = rng.standard_normal((L, 1, D))
    V = rng.standard_normal((L, 1, D))
    k, v, tbl = _single_seq(K, V, 16, perm_seed=4)
    q = rng.standard_normal((1, 1, D))
    out = oracle.decode_attention(q, k, v, tbl, [L], scale=0.0)
    np.testing.assert_allclose(out[0, 0], V[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    L, D = 20, 8
    K = np.repeat(rng.standard_normal((1, 1, D)), L, axis=0)
    V = rng.standard_normal((L, 1, D))
    k, v, tbl = _single_seq(K, V, 16, perm_seed=5)
    q = rng.standard_normal((1, 1, D))
    out = oracle.decode_attention(q, k, v, tbl, [L], scale=1.3)
    np.testing.assert_allclose(out[0, 0], V[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_two_token_logistic_closed_form():
    """q = e0, k0 = 2 e0, k1 = 0, scale 1/2: scores (1, 0), so the weights are
    e/(1+e) and 1/(1+e). Catches a dropped or inverted scale and a flipped sign."""
    q = np.array([[[1.0, 0, 0, 0]]])
    K = np.array([[[2.0, 0, 0, 0]], [[0.0, 0, 0, 0]]])
    V = np.array([[[1.0, 0, 0, 0]], [[0.0, 1, 0, 0]]])
    k, v, tbl = _single_seq(K, V, 16)
    out = oracle.decode_attention(q, k, v, tbl, [2], scale=0.5)
    w0 = math.e / (1.0 + math.e)
    np.testing.assert_allclose(out[0, 0], [w0, 1.0 - w0, 0, 0], rtol=0, atol=1e-15)


@pytest.mark.parametrize("j", [0, 5, 16, 17, 30])
def test_one_hot_key_closed_form(j):
    """K_t = e_t, q = c e_j: score c*scale at t = j and 0 elsewhere, so
    out = (e^{c s} V_j + sum_{t != j} V_t) / (e^{c s} + L - 1). A wrong block or
    offset index picks the wrong V row and fails."""
    L, D, bs = 31, 32, 16
    rng = np.random.default_rng(10 + j)
    K = np.zeros((L, 1, D))
    for t in range(L):
        K[t, 0, t] = 1.0
    V = rng.standard_normal((L, 1, D))
    k, v, tbl = _single_seq(K, V, bs, perm_seed=j)
    c, s = 12.0, 0.5
    q = np.zeros((1, 1, D))
    q[0, 0, j] = c
    out = oracle.decode_attention(q, k, v, tbl, [L], scale=s)
    a = math.exp(c * s)
    expect = (a * V[j, 0] + (V[:, 0].sum(axis=0) - V[j, 0])) / (a + L - 1)
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-13, atol=1e-14)


def test_empty_sequence_gives_zero():
    q, k, v, tables, lengths = _random_case(0)
    lengths = lengths.copy()
    lengths[1] = 0
    out = oracle.decode_attention(q, k, v, tables, lengths, 0.5)
    assert np.all(out[1] == 0)
    assert np.all(np.isfinite(out))


# ---------------------------------------------------------------------------
# Brute force: 50-digit arithmetic, walking the physical cache
# ---------------------------------------------------------------------------

def _brute_force(q, k, v, tables, lengths, scale, bs):
    """For every physical slot, find which (request, position) owns it by inverting the
    block tables, then form sum_t exp(z_t) V_t / sum_t exp(z_t) in mpmath (no max
    subtraction). Independent of the oracle's gather and of numpy's exp."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    B, Hq, D = q.shape
    NB, Hkv = k.shape[0], k.shape[1]
    g = Hq // Hkv
    owners = {}
    for s in range(B):
        n = -(-int(lengths[s]) // bs)
        for j in range(n):
            owners.setdefault(int(tables[s][j]), []).append((s, j))
    out = np.zeros((B, Hq, D))
    for s in range(B):
        for h in range(Hq):
            kvh = next(c for c in range(Hkv) if c * g <= h < (c + 1) * g)
            num = [mpmath.mpf(0)] * D
            den = mpmath.mpf(0)
            for phys in range(NB):
                for (s2, j) in owners.get(phys, []):
                    if s2 != s:
                        continue
                    for off in range(bs):
                        pos = j * bs + off
                        if pos >= int(lengths[s]):
                            continue
                        z = mpmath.mpf(0)
                        for d in range(D):
                            z += mpmath.mpf(float(q[s, h, d])) * mpmath.mpf(float(k[phys, kvh, off, d]))
                        e = mpmath.exp(mpmath.mpf(scale) * z)
                        den += e
                        for d in range(D):
                            num[d] += e * mpmath.mpf(float(v[phys, kvh, off, d]))
            if den > 0:
                out[s, h] = [float(x / den) for x in num]
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_matches_brute_force(seed):
    q, k, v, tables, lengths = _random_case(seed, B=2, Hq=4, Hkv=2, D=3, bs=4, max_len=9)
    scale = 0.7
    got = oracle.decode_attention(q, k, v, tables, lengths, scale)
    ref = _brute_force(q, k, v, tables, lengths, scale, 4)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def _relayout(k, v, tables, lengths, bs, perm):
    """Move every physical block b to perm[b] and rewrite the tables to match."""
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    t2 = np.array(tables, copy=True)
    for s in range(len(lengths)):
        n = -(-int(lengths[s]) // bs)
        t2[s, :n] = perm[tables[s, :n]]
    return k2, v2, t2


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_permutation_of_physical_blocks_is_invisible(seed):
    q, k, v, tables, lengths = _random_case(seed, B=4, Hq=6, Hkv=3, D=8, bs=4, max_len=30)
    perm = np.random.default_rng(100 + seed).permutation(k.shape[0])
    k2, v2, t2 = _relayout(k, v, tables, lengths, 4, perm)
    a = oracle.decode_attention(q, k, v, tables, lengths, 0.4)
    b = oracle.decode_attention(q, k2, v2, t2, lengths, 0.4)
    assert np.array_equal(a, b)


def test_shared_prefix_equals_private_copies():
    """Requests whose tables share refcounted prefix blocks give exactly the result
    of the same requests with private copies of those blocks."""
    rng = np.random.default_rng(7)
    bs, B, Hkv, Hq, D = 4, 5, 2, 4, 8
    prefix = 12
    lengths = prefix + rng.integers(1, 10, size=B)
    tables, _, NB, alloc = build_tables(lengths, bs, rng, shared_prefix_tokens=prefix)
    pre_blocks = tables[0, :prefix // bs]
    assert all(np.array_equal(tables[s, :prefix // bs], pre_blocks) for s in range(B))
    assert all(alloc.refcount[b] == B for b in pre_blocks)
    q = _bf16_exact(rng.standard_normal((B, Hq, D)))
    k = _bf16_exact(rng.standard_normal((NB, Hkv, bs, D)))
    v = _bf16_exact(rng.standard_normal((NB, Hkv, bs, D)))
    shared = oracle.decode_attention(q, k, v, tables, lengths, 0.3)
    # private layout: append (B-1) copies of the prefix blocks at the end of the pool
    npre = len(pre_blocks)
    k2 = np.concatenate([k] + [k[pre_blocks]] * (B - 1))
    v2 = np.concatenate([v] + [v[pre_blocks]] * (B - 1))
    t2 = np.array(tables, copy=True)
    for s in range(1, B):
        t2[s, :npre] = NB + (s - 1) * npre + np.arange(npre)
    private = oracle.decode_attention(q, k2, v2, t2, lengths, 0.3)
    assert np.array_equal(shared, private)


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(11)
    for L in (1, 2, 17, 300):
        K = rng.standard_normal((L, 16)) * 3
        V = rng.standard_normal((L, 16))
        q = rng.standard_normal(16) * 3
        _, w = oracle.attend_one_head(q, K, V, 0.25)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(w >= 0)


def test_gqa_equals_mha_with_repeated_kv():
    q, k, v, tables, lengths = _random_case(5, B=3, Hq=8, Hkv=2, D=8, bs=4, max_len=20)
    g = 4
    k_rep = np.repeat(k, g, axis=1)   # kv head c becomes heads c*g .. c*g+g-1
    v_rep = np.repeat(v, g, axis=1)
    gqa = oracle.decode_attention(q, k, v, tables, lengths, 0.5)
    mha = oracle.decode_attention(q, k_rep, v_rep, tables, lengths, 0.5)
    assert np.array_equal(gqa, mha)


def test_block_size_invariance():
    """The same logical KV paged with 16- or 32-token blocks gives identical output."""
    rng = np.random.default_rng(12)
    B, Hkv, Hq, D = 3, 2, 4, 8
    lengths = np.array([70, 1, 33])
    q = _bf16_exact(rng.standard_normal((B, Hq, D)))
    rows_k = [_bf16_exact(rng.standard_normal((L, Hkv, D))) for L in lengths]
    rows_v = [_bf16_exact(rng.standard_normal((L, Hkv, D))) for L in lengths]
    outs = []
    for bs in (16, 32):
        tables, _, NB, _ = build_tables(lengths, bs, np.random.default_rng(bs))
        k = np.zeros((NB, Hkv, bs, D))
        v = np.zeros((NB, Hkv, bs, D))
        for s, L in enumerate(lengths):
            for t in range(L):
                k[tables[s, t // bs], :, t % bs] = rows_k[s][t]
                v[tables[s, t // bs], :, t % bs] = rows_v[s][t]
        outs.append(oracle.decode_attention(q, k, v, tables, lengths, 0.35))
    assert np.array_equal(outs[0], outs[1])


def test_unused_slots_are_never_read():
    q, k, v, tables, lengths = _random_case(6, B=3, Hq=2, Hkv=2, D=4, bs=4, max_len=13)
    k = k.copy()
    v = v.copy()
    used = np.zeros(k.shape[:1] + k.shape[2:3], dtype=bool)
    for s, L in enumerate(lengths):
        for t in range(int(L)):
            used[tables[s, t // 4], t % 4] = True
    mask = np.broadcast_to(~used[:, None, :], k.shape[:3])
    k[mask] = np.nan
    v[mask] = np.nan
    out = oracle.decode_attention(q, k, v, tables, lengths, 0.5)
    assert np.all(np.isfinite(out))


# ---------------------------------------------------------------------------
# Append
# ---------------------------------------------------------------------------

def test_append_round_trip_and_skip():
    rng = np.random.default_rng(13)
    bs, Hkv, D = 16, 2, 8
    lengths = np.array([47, 200, 1])
    tables, last_slots, NB, _ = build_tables(lengths, bs, rng)
    k_cache = np.full((NB, Hkv, bs, D), -7.0)
    v_cache = np.full((NB, Hkv, bs, D), -9.0)
    new_k = rng.standard_normal((4, Hkv, D))
    new_v = rng.standard_normal((4, Hkv, D))
    slots = np.concatenate([last_slots, [-1]])
    k2, v2 = oracle.append_scatter(new_k, new_v, k_cache, v_cache, slots, bs)
    for s, L in enumerate(lengths):
        K = oracle.gather_sequence(k2, tables[s], L, 1, bs)
        assert np.array_equal(K[L - 1], new_k[s, 1])
        V = oracle.gather_sequence(v2, tables[s], L, 0, bs)
        assert np.array_equal(V[L - 1], new_v[s, 0])
    # exactly 3 token rows per head changed; the skipped token wrote nothing
    changed = np.any(k2 != k_cache, axis=-1)
    assert changed.sum() == 3 * Hkv
    assert np.all(v2[~np.any(v2 != v_cache, axis=-1)] == -9.0)


# ---------------------------------------------------------------------------
# INT8 quantiser
# ---------------------------------------------------------------------------

def test_quantizer_unit_scale_rounds_half_to_even():
    """absmax 127 makes s = 1 exactly, so q = rint(x): halves go to the even code."""
    x = np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 126.5, -127.0]], dtype=np.float32)
    q, s = oracle.quantize_rows_int8(x)
    assert s[0] == np.float32(1.0)
    assert q[0].tolist() == [127, 2, 4, -2, 0, 0, 126, -127]


def test_quantizer_zero_row():
    q, s = oracle.quantize_rows_int8(np.zeros((2, 5), dtype=np.float32))
    assert np.all(q == 0) and np.all(s == 0)


def test_quantizer_is_nearest_code_brute_force():
    """Against an exhaustive search over all 255 codes in fp32 (ties to even code)."""
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((6, 16)) * rng.uniform(0.01, 50, size=(6, 1))).astype(np.float32)
    x = _bf16_exact(x).astype(np.float32)
    q, s = oracle.quantize_rows_int8(x)
    codes = np.arange(-127, 128, dtype=np.float32)
    for r in range(x.shape[0]):
        assert s[r] == np.float32(np.max(np.abs(x[r]))) / np.float32(127)
        for c in range(x.shape[1]):
            ratio = np.float32(x[r, c] / s[r])
            dist = np.abs(codes - ratio)
            best = codes[dist == dist.min()]
            pick = best[0] if len(best) == 1 else best[np.argmin(np.abs(best) % 2)]
            assert q[r, c] == pick
        # the absmax element maps to +-127 and dequantisation error is <= s/2
        assert np.max(np.abs(q[r])) == 127
        err = np.abs(oracle.dequantize_rows_int8(q[r:r+1], s[r:r+1])[0] - x[r].astype(np.float64))
        assert np.all(err <= s[r] / 2 * (1 + 1e-6))


def test_int8_single_token_closed_form():
    """One token: the output is that token's dequantised V row (code x scale)."""
    D, bs = 8, 32
    kq = np.arange(-4, 4, dtype=np.int8).reshape(1, 1, 1, D).repeat(bs, axis=2)
    vq = np.arange(1, 9, dtype=np.int8).reshape(1, 1, 1, D).repeat(bs, axis=2)
    ks = np.full((1, 1, bs), 0.5, dtype=np.float32)
    vs = np.full((1, 1, bs), 0.03125, dtype=np.float32)
    q = np.ones((1, 1, D))
    out = oracle.decode_attention_int8(q, kq, vq, ks, vs, np.array([[0]]), [1], 0.1)
    assert np.array_equal(out[0, 0], np.arange(1, 9) * 0.03125)


def test_int8_append_then_decode_matches_dequantised_bf16_path():
    rng = np.random.default_rng(15)
    bs, Hkv, Hq, D = 16, 2, 4, 8
    lengths = np.array([5, 16, 17])
    tables, _, NB, _ = build_tables(lengths, bs, rng)
    kc = np.zeros((NB, Hkv, bs, D), dtype=np.int8)
    vc = np.zeros((NB, Hkv, bs, D), dtype=np.int8)
    ksc = np.zeros((NB, Hkv, bs), dtype=np.float32)
    vsc = np.zeros((NB, Hkv, bs), dtype=np.float32)
    # append every token of every request through the quantising scatter
    for s, L in enumerate(lengths):
        slots = [tables[s, t // bs] * bs + t % bs for t in range(L)]
        kk = _bf16_exact(rng.standard_normal((L, Hkv, D))).astype(np.float32)
        vv = _bf16_exact(rng.standard_normal((L, Hkv, D))).astype(np.float32)
        kc, vc, ksc, vsc = oracle.append_scatter_int8(kk, vv, kc, vc, ksc, vsc, slots, bs)
    q = _bf16_exact(rng.standard_normal((3, Hq, D)))
    a = oracle.decode_attention_int8(q, kc, vc, ksc, vsc, tables, lengths, 0.3)
    kr = oracle.dequantize_rows_int8(kc, ksc)
    vr = oracle.dequantize_rows_int8(vc, vsc)
    b = oracle.decode_attention(q, kr, vr, tables, lengths, 0.3)
    assert np.array_equal(a, b)


def test_int8_append_places_codes_and_scales_at_each_slot():
    """Read-back through the block tables (block manager of the chenk.top page, "块管理器：
    分页如何运作"; slot = block * block_size + offset): token t of sequence s is found in
    block tables[s, t // bs] at offset t % bs, its K codes and K scale in the K arrays
    and its V codes and V scale in the V arrays, and each row dequantises to within half
    a step (s / 2) of the row that was appended. A token with slot -1 writes nothing, and
    every slot no token was given keeps the canary it held before."""
    rng = np.random.default_rng(17)
    bs, Hkv, D = 16, 2, 8
    lengths = np.array([5, 16, 17, 40])
    tables, _, NB, _ = build_tables(lengths, bs, rng)
    NB += 1                                # block NB - 1 (index -1) is never in a table
    canary_code, canary_scale = 99, np.float32(-7.0)
    kc = np.full((NB, Hkv, bs, D), canary_code, dtype=np.int8)
    vc = np.full((NB, Hkv, bs, D), -canary_code, dtype=np.int8)
    ksc = np.full((NB, Hkv, bs), canary_scale, dtype=np.float32)
    vsc = np.full((NB, Hkv, bs), canary_scale, dtype=np.float32)
    written = np.zeros((NB, bs), dtype=bool)
    rows = {}
    for s, L in enumerate(lengths):
        slots = [int(tables[s, t // bs]) * bs + t % bs for t in range(L)] + [-1]
        # K and V of different magnitudes, so that a K/V mix-up shows in the read-back
        kk = _bf16_exact(rng.standard_normal((L + 1, Hkv, D)) * 5.0).astype(np.float32)
        vv = _bf16_exact(rng.standard_normal((L + 1, Hkv, D)) * 0.25).astype(np.float32)
        kk[L] = 1000.0                     # the skipped token: a row no slot may receive
        vv[L] = -1000.0
        kc, vc, ksc, vsc = oracle.append_scatter_int8(kk, vv, kc, vc, ksc, vsc, slots, bs)
        for t in range(L):
            rows[(s, t)] = (kk[t], vv[t])
            written[tables[s, t // bs], t % bs] = True
    for (s, t), (k_row, v_row) in rows.items():
        blk, off = int(tables[s, t // bs]), t % bs
        for h in range(Hkv):
            for codes, scales, x in ((kc, ksc, k_row[h]), (vc, vsc, v_row[h])):
                sc = float(scales[blk, h, off])
                amax = float(np.max(np.abs(x)))
                # the scale belongs to this row: absmax / 127 within fp32 rounding
                assert abs(sc * 127.0 - amax) <= amax * 1e-6
                back = codes[blk, h, off].astype(np.float64) * sc
                # half a step, plus the fp32 rounding of x / s (a ratio up to 127)
                assert np.all(np.abs(back - x) <= sc * (0.5 + 1e-5))
                assert np.max(np.abs(codes[blk, h, off].astype(np.int64))) == 127
    # untouched slots keep their canaries (nothing of the skipped token landed anywhere)
    for blk in range(NB):
        for off in range(bs):
            if written[blk, off]:
                continue
            assert np.all(kc[blk, :, off] == canary_code)
            assert np.all(vc[blk, :, off] == -canary_code)
            assert np.all(ksc[blk, :, off] == canary_scale)
            assert np.all(vsc[blk, :, off] == canary_scale)


# ---------------------------------------------------------------------------
# Planted mistakes: every one must be caught by a pin above
# ---------------------------------------------------------------------------

def _plant(monkeypatch, name, fn):
    """Replace an oracle function both in its module and in the package namespace."""
    monkeypatch.setattr(pa, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def _fails(fn, *args):
    """True when the pin does not pass: an assertion or any error (such as reading a
    poison table entry) counts as the mistake being caught."""
    try:
        fn(*args)
    except Exception:
        return True
    return False


def test_pins_catch_wrong_kv_head_mapping(monkeypatch):
    # interleaved grouping (h % num_kv_heads) instead of consecutive (h // g); the
    # test case has 8 query heads
    _plant(monkeypatch, "_kv_head_of", lambda h, g: h % (8 // g) if g > 1 else h)
    assert _fails(test_gqa_equals_mha_with_repeated_kv)


def test_pins_catch_gather_ignoring_block_table(monkeypatch):
    def bad_gather(cache, row, L, kvh, bs):
        rows = [np.asarray(cache[t // bs, kvh, t % bs], dtype=np.float64) for t in range(int(L))]
        return np.stack(rows) if rows else np.zeros((0, cache.shape[-1]))
    _plant(monkeypatch, "gather_sequence", bad_gather)
    assert _fails(test_one_hot_key_closed_form, 17)
    assert _fails(test_permutation_of_physical_blocks_is_invisible, 0)


def test_pins_catch_swapped_block_and_offset(monkeypatch):
    def bad_gather(cache, row, L, kvh, bs):
        rows = [np.asarray(cache[int(row[t % bs]) if t % bs < len(row) else 0, kvh, t // bs],
                           dtype=np.float64) for t in range(int(L))]
        return np.stack(rows) if rows else np.zeros((0, cache.shape[-1]))
    _plant(monkeypatch, "gather_sequence", bad_gather)
    assert _fails(test_paging_worked_example_gather_reads_only_table_prefix)


def test_pins_catch_missing_scale_and_sign(monkeypatch):
    orig = pa.attend_one_head

    def no_scale(q, K, V, scale):
        return orig(q, K, V, 1.0)

    def neg(q, K, V, scale):
        return orig(q, K, V, -scale)
    _plant(monkeypatch, "attend_one_head", no_scale)
    assert _fails(test_two_token_logistic_closed_form)
    _plant(monkeypatch, "attend_one_head", neg)
    assert _fails(test_two_token_logistic_closed_form)


def test_pins_catch_off_by_one_length(monkeypatch):
    orig = pa.gather_sequence
    _plant(monkeypatch, "gather_sequence",
                        lambda c, r, L, h, bs: orig(c, r, max(int(L) - 1, 0), h, bs))
    assert _fails(test_zero_scale_gives_mean_of_values)


def test_pins_catch_round_half_away_from_zero(monkeypatch):
    def away(x):
        return np.sign(x) * np.floor(np.abs(x) + 0.5)
    monkeypatch.setattr(np, "rint", away)
    assert _fails(test_quantizer_unit_scale_rounds_half_to_even)


def _planted_int8_scatter(swap_kv=False, shift=0):
    """append_scatter_int8 with a mistake in where rows land: K and V swapped, or the
    offset inside the block moved by `shift`."""
    def scatter(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, block_size):
        kq, ks = pa.quantize_rows_int8(k)
        vq, vs = pa.quantize_rows_int8(v)
        kc, vc, ksc, vsc = [np.array(a, copy=True) for a in (k_cache, v_cache, k_scale, v_scale)]
        if swap_kv:
            kq, vq, ks, vs = vq, kq, vs, ks
        for t in range(len(slot_mapping)):
            slot = int(slot_mapping[t])
            if slot < 0:
                continue
            blk, off = slot // block_size, (slot + shift) % block_size
            kc[blk, :, off], vc[blk, :, off] = kq[t], vq[t]
            ksc[blk, :, off], vsc[blk, :, off] = ks[t], vs[t]
        return kc, vc, ksc, vsc
    return scatter


def test_pins_catch_int8_scatter_misplacement(monkeypatch):
    _plant(monkeypatch, "append_scatter_int8", _planted_int8_scatter(swap_kv=True))
    assert _fails(test_int8_append_places_codes_and_scales_at_each_slot)
    _plant(monkeypatch, "append_scatter_int8", _planted_int8_scatter(shift=1))
    assert _fails(test_int8_append_places_codes_and_scales_at_each_slot)
    # a scatter that writes the skipped token (slot -1 read as the last slot of the pool)
    orig = pa.append_scatter_int8

    def no_skip(k, v, kc, vc, ks, vs, slots, bs):
        nb = np.shape(kc)[0]
        slots = [int(x) if int(x) >= 0 else nb * bs - 1 for x in slots]
        return orig(k, v, kc, vc, ks, vs, slots, bs)
    _plant(monkeypatch, "append_scatter_int8", no_skip)
    assert _fails(test_int8_append_places_codes_and_scales_at_each_slot)
