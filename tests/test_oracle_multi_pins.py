"""Pins for the oracle's multi-query paged attention (q_len = k + 1 new tokens per
sequence, each attending causally; the verification pass of "推测解码" on the
chenk.top page).

Each check ties it to something other than itself: the single-query oracle (already
pinned by brute force and closed forms) on truncated contexts, closed forms that fix
the causal offset, brute force in 50-digit arithmetic over physical slots, and the
block-placement invariant. The last group plants mistakes and checks they are caught.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import paged_attention as pa
from paged_kv_decode_02_gb300.workloads import build_tables


def _case(seed, B=3, n=3, Hq=4, Hkv=2, D=4, bs=4, max_len=13):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(n, max_len + 1, size=B)
    lengths[-1] = 0                                   # an empty sequence
    tables, _, NB, _ = build_tables(lengths, bs, rng)
    q = rng.standard_normal((B, n, Hq, D))
    k = rng.standard_normal((NB, Hkv, bs, D))
    v = rng.standard_normal((NB, Hkv, bs, D))
    return q, k, v, tables, lengths


def test_single_query_is_decode_attention():
    q, k, v, tables, lengths = _case(0, n=1)
    a = oracle.decode_attention_multi(q, k, v, tables, lengths, 0.4)
    b = oracle.decode_attention(q[:, 0], k, v, tables, lengths, 0.4)
    assert np.array_equal(a[:, 0], b)


@pytest.mark.parametrize("seed", [1, 2])
def test_each_query_is_decode_over_its_causal_prefix(seed):
    n = 4
    q, k, v, tables, lengths = _case(seed, n=n)
    a = oracle.decode_attention_multi(q, k, v, tables, lengths, 0.3)
    for i in range(n):
        lens_i = np.where(lengths > 0, lengths - n + i + 1, 0)
        b = oracle.decode_attention(q[:, i], k, v, tables, lens_i, 0.3)
        assert np.array_equal(a[:, i], b)


def test_scale_zero_gives_running_means():
    """Context = exactly the q_len new tokens, scale 0: query i averages V[0..i]."""
    n, D, bs = 5, 3, 4
    rng = np.random.default_rng(3)
    tables, _, NB, _ = build_tables([n], bs, rng)
    v = rng.standard_normal((NB, 1, bs, D))
    k = rng.standard_normal((NB, 1, bs, D))
    q = rng.standard_normal((1, n, 1, D))
    out = oracle.decode_attention_multi(q, k, v, tables, [n], 0.0)
    V = np.stack([v[tables[0, t // bs], 0, t % bs] for t in range(n)])
    for i in range(n):
        assert np.allclose(out[0, i, 0], V[:i + 1].mean(axis=0), rtol=0, atol=1e-15)


def test_self_attending_keys_closed_form():
    """L = q_len = 3, K = 30 * I, q_i = e_i, scale 1: query i scores 30 on itself and
    0 on each of the i earlier tokens (later ones are invisible), so
    out_i = (e^30 V_i + sum_{j<i} V_j) / (e^30 + i)."""
    n, D, bs = 3, 4, 4
    rng = np.random.default_rng(4)
    tables = np.array([[0]])
    k = np.zeros((1, 1, bs, D))
    v = np.zeros((1, 1, bs, D))
    for t in range(n):
        k[0, 0, t, t] = 30.0
        v[0, 0, t] = rng.standard_normal(D)
    q = np.zeros((1, n, 1, D))
    for i in range(n):
        q[0, i, 0, i] = 1.0
    out = oracle.decode_attention_multi(q, k, v, tables, [n], 1.0)
    E = math.exp(30.0)
    for i in range(n):
        want = (E * v[0, 0, i] + v[0, 0, :i].sum(axis=0)) / (E + i)
        assert np.allclose(out[0, i, 0], want, rtol=1e-13, atol=0)


def _brute(q, k, v, tables, lengths, scale, bs):
    """50-digit brute force: every physical slot, owner and position from the inverted
    tables, causal visibility from positions, no max subtraction."""
    import mpmath
    mpmath.mp.dps = 50
    B, n, Hq, D = q.shape
    NB, Hkv = k.shape[0], k.shape[1]
    g = Hq // Hkv
    out = np.zeros(q.shape)
    for s in range(B):
        L = int(lengths[s])
        if L == 0:
            continue
        pos_of = {}
        for j in range(-(-L // bs)):
            for o in range(bs):
                if j * bs + o < L:
                    pos_of[(int(tables[s, j]), o)] = j * bs + o
        for i in range(n):
            for h in range(Hq):
                num = [mpmath.mpf(0)] * D
                den = mpmath.mpf(0)
                for blk in range(NB):
                    for o in range(bs):
                        t = pos_of.get((blk, o))
                        if t is None or t > L - n + i:
                            continue
                        z = mpmath.mpf(0)
                        for d in range(D):
                            z += mpmath.mpf(float(q[s, i, h, d])) * mpmath.mpf(float(k[blk, h // g, o, d]))
                        e = mpmath.exp(mpmath.mpf(scale) * z)
                        den += e
                        for d in range(D):
                            num[d] += e * mpmath.mpf(float(v[blk, h // g, o, d]))
                out[s, i, h] = [float(x / den) for x in num]
    return out


def test_matches_brute_force():
    q, k, v, tables, lengths = _case(5, B=2, n=3, max_len=9)
    a = oracle.decode_attention_multi(q, k, v, tables, lengths, 0.7)
    b = _brute(q, k, v, tables, lengths, 0.7, 4)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_block_placement_is_invisible():
    q, k, v, tables, lengths = _case(6, n=2)
    a = oracle.decode_attention_multi(q, k, v, tables, lengths, 0.5)
    rng = np.random.default_rng(7)
    NB = k.shape[0]
    perm = rng.permutation(NB)          # new physical id of each block
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm], v2[perm] = k, v
    t2 = np.where(tables >= 0, perm[np.clip(tables, 0, NB - 1)], tables)
    b = oracle.decode_attention_multi(q, k2, v2, t2, lengths, 0.5)
    assert np.array_equal(a, b)


def _quantized_case(seed, fmt, n=3, B=3, Hq=4, Hkv=2, D=8, bs=4, max_len=13):
    """Random codes and scales of a one-byte cache, with the dequantised real values."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(n, max_len + 1, size=B)
    lengths[-1] = 0
    tables, _, NB, _ = build_tables(lengths, bs, rng)
    if fmt == "int8":
        kc = rng.integers(-127, 128, size=(NB, Hkv, bs, D)).astype(np.int8)
        vc = rng.integers(-127, 128, size=(NB, Hkv, bs, D)).astype(np.int8)
        deq = lambda c, sc: oracle.dequantize_rows_int8(c, sc)  # noqa: E731
    else:
        finite = np.flatnonzero(np.isfinite(oracle.fp8_decode(np.arange(256), fmt)))
        kc = rng.choice(finite, size=(NB, Hkv, bs, D)).astype(np.uint8)
        vc = rng.choice(finite, size=(NB, Hkv, bs, D)).astype(np.uint8)
        deq = lambda c, sc: oracle.dequantize_rows_fp8(c, sc, fmt)  # noqa: E731
    ks = rng.uniform(0.005, 0.03, size=(NB, Hkv, bs)).astype(np.float32)
    vs = rng.uniform(0.005, 0.03, size=(NB, Hkv, bs)).astype(np.float32)
    q = rng.standard_normal((B, n, Hq, D))
    return q, kc, vc, ks, vs, deq(kc, ks), deq(vc, vs), tables, lengths


@pytest.mark.parametrize("fmt", ["int8", "e4m3", "e5m2"])
def test_quantized_equals_multi_on_dequantised_values(fmt):
    """Over a one-byte cache the multi-query oracle is the (pinned) multi-query oracle
    on the dequantised values: code x scale, decoded exactly."""
    q, kc, vc, ks, vs, kr, vr, tables, lengths = _quantized_case(20, fmt)
    a = oracle.decode_attention_multi_quantized(q, kc, vc, ks, vs, tables, lengths, 0.3, fmt)
    b = oracle.decode_attention_multi(q, kr, vr, tables, lengths, 0.3)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_quantized_single_query_is_single_token_decode(fmt):
    """q_len = 1 over a one-byte cache is the (pinned) single-token INT8 / FP8 oracle."""
    q, kc, vc, ks, vs, _, _, tables, lengths = _quantized_case(21, fmt, n=1)
    a = oracle.decode_attention_multi_quantized(q, kc, vc, ks, vs, tables, lengths, 0.4, fmt)
    if fmt == "int8":
        b = oracle.decode_attention_int8(q[:, 0], kc, vc, ks, vs, tables, lengths, 0.4)
    else:
        b = oracle.decode_attention_fp8(q[:, 0], kc, vc, ks, vs, tables, lengths, 0.4, fmt)
    assert np.array_equal(a[:, 0], b)


def test_quantized_closed_form_running_means():
    """Scale 0, context = the q_len new tokens: query i averages code x scale of V rows
    0..i (the scales multiply the V codes, the K codes do not matter)."""
    n, D, bs = 4, 3, 4
    rng = np.random.default_rng(22)
    tables, _, NB, _ = build_tables([n], bs, rng)
    vc = rng.integers(-127, 128, size=(NB, 1, bs, D)).astype(np.int8)
    kc = rng.integers(-127, 128, size=(NB, 1, bs, D)).astype(np.int8)
    vs = rng.uniform(0.01, 0.02, size=(NB, 1, bs)).astype(np.float32)
    ks = rng.uniform(0.01, 0.02, size=(NB, 1, bs)).astype(np.float32)
    out = oracle.decode_attention_multi_quantized(rng.standard_normal((1, n, 1, D)), kc, vc,
                                                  ks, vs, tables, [n], 0.0, "int8")
    vals = [vc[tables[0, t // bs], 0, t % bs].astype(np.float64) *
            float(vs[tables[0, t // bs], 0, t % bs]) for t in range(n)]
    for i in range(n):
        assert np.allclose(out[0, i, 0], np.mean(vals[:i + 1], axis=0), rtol=0, atol=1e-15)


def test_too_short_context_is_refused():
    q = np.zeros((1, 3, 1, 2))
    with pytest.raises(ValueError):
        oracle.decode_attention_multi(q, np.zeros((1, 1, 4, 2)), np.zeros((1, 1, 4, 2)),
                                      np.array([[0]]), [2], 1.0)


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _fails(fn, *args):
    try:
        fn(*args)
    except Exception:
        return True
    return False


def _plant_visible(monkeypatch, visible_of):
    """Replace the oracle's causal window: visible_of(L, n, i) -> tokens seen."""
    def bad(q, k_cache, v_cache, block_tables, context_lens, scale, block_size=None):
        q = np.asarray(q)
        B, n, Hq, D = q.shape
        Hkv = k_cache.shape[1]
        bs = block_size or k_cache.shape[2]
        g = Hq // Hkv
        out = np.zeros((B, n, Hq, D))
        for s in range(B):
            L = int(context_lens[s])
            if L == 0:
                continue
            for kvh in range(Hkv):
                K = pa.gather_sequence(k_cache, block_tables[s], L, kvh, bs)
                V = pa.gather_sequence(v_cache, block_tables[s], L, kvh, bs)
                for i in range(n):
                    m = max(0, min(L, visible_of(L, n, i)))
                    for h in range(kvh * g, (kvh + 1) * g):
                        out[s, i, h], _ = pa.attend_one_head(q[s, i, h], K[:m], V[:m], scale)
        return out
    monkeypatch.setattr(pa, "decode_attention_multi", bad)
    monkeypatch.setattr(oracle, "decode_attention_multi", bad)


def test_pins_catch_off_by_one_window(monkeypatch):
    _plant_visible(monkeypatch, lambda L, n, i: L - n + i)
    assert _fails(test_scale_zero_gives_running_means)
    assert _fails(test_each_query_is_decode_over_its_causal_prefix, 1)


def test_pins_catch_missing_causal_mask(monkeypatch):
    _plant_visible(monkeypatch, lambda L, n, i: L)
    assert _fails(test_self_attending_keys_closed_form)
    assert _fails(test_matches_brute_force)


def test_pins_catch_reversed_query_order(monkeypatch):
    _plant_visible(monkeypatch, lambda L, n, i: L - i)
    assert _fails(test_scale_zero_gives_running_means)


def _plant_quantized(monkeypatch, swap_scales=False, visible_of=None):
    """Replace the one-byte multi-query oracle by one with a mistake: K and V scales
    exchanged, or another causal window visible_of(L, n, i)."""
    def bad(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale, fmt,
            block_size=None):
        q = np.asarray(q)
        B, n, Hq, D = q.shape
        Hkv = k_codes.shape[1]
        bs = block_size or k_codes.shape[2]
        g = Hq // Hkv
        ks, vs = (v_scale, k_scale) if swap_scales else (k_scale, v_scale)
        out = np.zeros((B, n, Hq, D))
        for s in range(B):
            L = int(context_lens[s])
            if L == 0:
                continue
            for kvh in range(Hkv):
                K = pa.gather_sequence_int8(k_codes, ks, block_tables[s], L, kvh, bs)
                V = pa.gather_sequence_int8(v_codes, vs, block_tables[s], L, kvh, bs)
                for i in range(n):
                    m = L - n + i + 1 if visible_of is None else visible_of(L, n, i)
                    m = max(0, min(L, m))
                    for h in range(kvh * g, (kvh + 1) * g):
                        out[s, i, h], _ = pa.attend_one_head(q[s, i, h], K[:m], V[:m], scale)
        return out
    monkeypatch.setattr(pa, "decode_attention_multi_quantized", bad)
    monkeypatch.setattr(oracle, "decode_attention_multi_quantized", bad)


def test_pins_catch_quantized_scales_swapped(monkeypatch):
    _plant_quantized(monkeypatch, swap_scales=True)
    assert _fails(test_quantized_closed_form_running_means)
    assert _fails(test_quantized_equals_multi_on_dequantised_values, "int8")


def test_pins_catch_quantized_missing_causal_window(monkeypatch):
    _plant_quantized(monkeypatch, visible_of=lambda L, n, i: L)
    assert _fails(test_quantized_equals_multi_on_dequantised_values, "int8")
    assert _fails(test_quantized_closed_form_running_means)
