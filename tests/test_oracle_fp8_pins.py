"""Pins for the oracle's FP8 KV-cache functions (E4M3 and E5M2 codes with per-token
scales; "FP8（及 H100/H200 硬件路径）" and "KV 缓存量化" of the chenk.top page).

Each check ties the oracle to something other than itself: PyTorch's own float8
dtypes (a separate implementation of both formats), IEEE binary16 as numpy decodes
it (an E5M2 code is the upper byte of a binary16), exhaustive search over every
finite code, the format's defining constants, and reductions to the pinned bf16
attention. The last group plants mistakes in the oracle and checks they are caught.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_decode_02_gb300.workloads import build_tables

FMTS = ("e4m3", "e5m2")
TORCH_DT = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _bf16_exact(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _torch_codes(x, fmt):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(TORCH_DT[fmt]) \
        .view(torch.uint8).numpy()


def _same_values(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and \
        np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


# ---------------------------------------------------------------------------
# Decoding
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
def test_decode_matches_torch_float8_for_every_code(fmt):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(TORCH_DT[fmt]).double().numpy()
    assert _same_values(oracle.fp8_decode(np.arange(256), fmt), ref)


def test_e5m2_code_is_the_upper_byte_of_binary16():
    c = np.arange(256, dtype=np.uint16)
    ref = (c << 8).astype(np.uint16).view(np.float16).astype(np.float64)
    assert _same_values(oracle.fp8_decode(c, "e5m2"), ref)


def test_e4m3_is_binary16_with_the_exponent_rebiased():
    """S.EEEE.MMM placed as binary16 S.0EEEE.MMM0000000 is the value times 2^-8 (biases
    7 and 15), subnormals included; the single NaN pattern aside."""
    c = np.arange(256, dtype=np.uint16)
    h = ((c & 0x80) << 8) | ((c & 0x7F) << 7)
    ref = h.astype(np.uint16).view(np.float16).astype(np.float64) * 256.0
    mine = oracle.fp8_decode(c, "e4m3")
    nan = (c & 0x7F) == 0x7F
    assert np.all(np.isnan(mine[nan]))
    assert np.array_equal(mine[~nan], ref[~nan])


def test_format_constants():
    d = lambda c, f: float(oracle.fp8_decode([c], f)[0])  # noqa: E731
    # E4M3: bias 7, largest finite 448 = 1.75 * 2^8, no infinity
    assert d(0x38, "e4m3") == 1.0 and d(0x7E, "e4m3") == 448.0
    assert d(0x08, "e4m3") == 2.0 ** -6 and d(0x01, "e4m3") == 2.0 ** -9
    assert not np.any(np.isinf(oracle.fp8_decode(np.arange(256), "e4m3")))
    assert oracle.FP8_MAX["e4m3"] == 448.0
    # E5M2: bias 15, largest finite 57344 = 1.75 * 2^15, infinities at 0x7C / 0xFC
    assert d(0x3C, "e5m2") == 1.0 and d(0x7B, "e5m2") == 57344.0
    assert d(0x04, "e5m2") == 2.0 ** -14 and d(0x01, "e5m2") == 2.0 ** -16
    assert d(0x7C, "e5m2") == np.inf and d(0xFC, "e5m2") == -np.inf
    assert oracle.FP8_MAX["e5m2"] == 57344.0
    # E5M2 trades precision for range: a wider span, a coarser step near 1
    assert oracle.FP8_MAX["e5m2"] > oracle.FP8_MAX["e4m3"]
    assert d(0x39, "e4m3") - 1.0 == 0.125 and d(0x3D, "e5m2") - 1.0 == 0.25


# ---------------------------------------------------------------------------
# Rounding and the per-row quantiser
# ---------------------------------------------------------------------------

def _probe_values(fmt, seed):
    rng = np.random.default_rng(seed)
    mags = rng.choice([1e-5, 1e-3, 3e-2, 1.0, 30.0, 300.0, 20000.0], 4000)
    x = (rng.standard_normal(4000) * mags).astype(np.float32)
    # exact midpoints between neighbouring codes (ties) and the codes themselves
    vals = oracle.fp8_decode(np.arange(0, 127), fmt)
    vals = vals[np.isfinite(vals)]
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, vals.astype(np.float32)])
    return x[np.abs(x) <= oracle.FP8_MAX[fmt]]


@pytest.mark.parametrize("fmt", FMTS)
def test_round_matches_torch_float8_in_range(fmt):
    x = _probe_values(fmt, 3)
    assert np.array_equal(oracle.fp8_round(x, fmt), _torch_codes(x, fmt))


@pytest.mark.parametrize("fmt", FMTS)
def test_round_is_nearest_code_ties_even_brute_force(fmt):
    x = _probe_values(fmt, 4)[::7]
    got = oracle.fp8_round(x, fmt)
    codes = np.arange(256)
    allv = oracle.fp8_decode(codes, fmt)
    fin = np.isfinite(allv)
    for xi, c in zip(x.astype(np.float64), got):
        dist = np.abs(allv[fin] - xi)
        best = codes[fin][dist == dist.min()]
        assert abs(float(oracle.fp8_decode([c], fmt)[0]) - xi) == dist.min()
        if len(best) > 1 and np.any(oracle.fp8_decode(best, fmt) != 0):
            assert c % 2 == 0          # a tie between two codes goes to the even one


@pytest.mark.parametrize("fmt", FMTS)
def test_round_saturates_to_the_largest_finite_code(fmt):
    big = np.array([1e9, -1e9, oracle.FP8_MAX[fmt] * 1.2, -oracle.FP8_MAX[fmt] * 1.01],
                   dtype=np.float32)
    top = 0x7E if fmt == "e4m3" else 0x7B
    assert oracle.fp8_round(big, fmt).tolist() == [top, top | 0x80, top, top | 0x80]


@pytest.mark.parametrize("fmt", FMTS)
def test_quantizer_rows(fmt):
    rng = np.random.default_rng(5)
    x = _bf16_exact(rng.standard_normal((8, 64)) * rng.uniform(0.01, 80, (8, 1))) \
        .astype(np.float32)
    x[3] = 0.0
    q, s = oracle.quantize_rows_fp8(x, fmt)
    top = 0x7E if fmt == "e4m3" else 0x7B
    for r in range(8):
        amax = np.float32(np.max(np.abs(x[r])))
        assert s[r] == amax / np.float32(oracle.FP8_MAX[fmt])
        if amax == 0:
            assert np.all(q[r] == 0)
            continue
        # the absmax element takes the largest code; the rest round to nearest
        assert np.max(q[r] & 0x7F) == top
        ratio = (x[r] / s[r]).astype(np.float32)
        assert np.array_equal(q[r], _torch_codes(ratio, fmt))
        # error bound: half a step of the code's binade, or of the subnormal step
        err = np.abs(oracle.dequantize_rows_fp8(q[r:r+1], s[r:r+1], fmt)[0] - x[r])
        mbits = 3 if fmt == "e4m3" else 2
        sub = 2.0 ** (-6 - 3) if fmt == "e4m3" else 2.0 ** (-14 - 2)
        bound = np.maximum(np.abs(x[r]) * 2.0 ** -(mbits + 1), sub / 2 * float(s[r]))
        assert np.all(err <= bound * (1 + 1e-6))


# ---------------------------------------------------------------------------
# FP8 attention
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
def test_single_token_closed_form(fmt):
    """One token: the output is its decoded V row times its scale."""
    D, bs = 8, 16
    codes = np.array([0x38, 0x40, 0xB8, 0x00, 0x30, 0x44, 0x3C, 0x3A], dtype=np.uint8)
    kq = np.zeros((1, 1, bs, D), dtype=np.uint8)
    vq = np.broadcast_to(codes, (1, 1, bs, D)).copy()
    ks = np.full((1, 1, bs), 0.5, dtype=np.float32)
    vs = np.full((1, 1, bs), 0.25, dtype=np.float32)
    out = oracle.decode_attention_fp8(np.ones((1, 1, D)), kq, vq, ks, vs, np.array([[0]]), [1],
                                      0.1, fmt)
    assert np.array_equal(out[0, 0], oracle.fp8_decode(codes, fmt) * 0.25)


@pytest.mark.parametrize("fmt", FMTS)
def test_append_then_decode_matches_dequantised_bf16_path(fmt):
    rng = np.random.default_rng(16)
    bs, Hkv, Hq, D = 16, 2, 8, 8
    lengths = np.array([5, 16, 17, 40])
    tables, _, NB, _ = build_tables(lengths, bs, rng)
    kc = np.zeros((NB, Hkv, bs, D), dtype=np.uint8)
    vc = np.zeros((NB, Hkv, bs, D), dtype=np.uint8)
    ksc = np.zeros((NB, Hkv, bs), dtype=np.float32)
    vsc = np.zeros((NB, Hkv, bs), dtype=np.float32)
    for s, L in enumerate(lengths):
        slots = [tables[s, t // bs] * bs + t % bs for t in range(L)]
        kk = _bf16_exact(rng.standard_normal((L, Hkv, D)) * 3).astype(np.float32)
        vv = _bf16_exact(rng.standard_normal((L, Hkv, D))).astype(np.float32)
        kc, vc, ksc, vsc = oracle.append_scatter_fp8(kk, vv, kc, vc, ksc, vsc, slots, bs, fmt)
        # each appended row reads back within the quantiser's bound
        for t in range(L):
            blk, off = tables[s, t // bs], t % bs
            back = oracle.fp8_decode(kc[blk, :, off], fmt) * ksc[blk, :, off, None]
            assert np.all(np.abs(back - kk[t]) <= np.abs(kk[t]).max(-1, keepdims=True) * 0.14)
    q = _bf16_exact(rng.standard_normal((len(lengths), Hq, D)))
    a = oracle.decode_attention_fp8(q, kc, vc, ksc, vsc, tables, lengths, 0.3, fmt)
    kr = oracle.dequantize_rows_fp8(kc, ksc, fmt)
    vr = oracle.dequantize_rows_fp8(vc, vsc, fmt)
    b = oracle.decode_attention(q, kr, vr, tables, lengths, 0.3)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _plant(monkeypatch, name, fn):
    monkeypatch.setattr(pa, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def _fails(fn, *args):
    try:
        fn(*args)
    except Exception:
        return True
    return False


def test_pins_catch_wrong_exponent_bias(monkeypatch):
    monkeypatch.setitem(pa.FP8_FORMATS, "e4m3", (4, 3, 8))
    assert _fails(test_decode_matches_torch_float8_for_every_code, "e4m3")
    assert _fails(test_format_constants)


def test_pins_catch_swapped_exponent_and_mantissa_widths(monkeypatch):
    monkeypatch.setitem(pa.FP8_FORMATS, "e5m2", (4, 3, 15))
    assert _fails(test_e5m2_code_is_the_upper_byte_of_binary16)


def test_pins_catch_ties_away_from_zero(monkeypatch):
    orig = pa.fp8_round

    def away(x, fmt):
        x = np.asarray(x, dtype=np.float32)
        nudged = np.nextafter(np.abs(x), np.float32(np.inf)) * np.sign(x)
        return orig(nudged.astype(np.float32), fmt)
    _plant(monkeypatch, "fp8_round", away)
    assert _fails(test_round_matches_torch_float8_in_range, "e4m3")


def test_pins_catch_missing_scale(monkeypatch):
    orig = pa.gather_sequence_fp8
    _plant(monkeypatch, "gather_sequence_fp8",
           lambda c, s, r, L, h, bs, f: orig(c, np.ones_like(s), r, L, h, bs, f))
    assert _fails(test_single_token_closed_form, "e5m2")


def test_pins_catch_scale_from_wrong_maximum(monkeypatch):
    monkeypatch.setitem(pa.FP8_MAX, "e4m3", 240.0)
    assert _fails(test_quantizer_rows, "e4m3")
