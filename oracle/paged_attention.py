"""fp64 CPU oracle for paged-KV append and single-token decode attention.

TEST INFRASTRUCTURE: imported only by tests, the smoke check and the CPU-baseline leg
of the benchmark. Nothing in the product library calls it.

Readings of the pages that this file fixes (the pages leave them open):

* Cache layout: K and V are separate arrays shaped ``[num_blocks, num_kv_heads,
  block_size, head_dim]``. Only the addressing matters for the result, so any layout
  read through the same indexing gives the same output.
* Slot encoding: ``slot = physical_block * block_size + offset``; a negative slot
  means "no token" and is skipped.
* Grouped-query attention: query head ``h`` reads KV head ``h // g`` with
  ``g = num_q_heads // num_kv_heads`` (consecutive grouping).
* ``context_lens[s]`` counts every cached token the new query attends to, the token
  appended in this step included; a sequence with 0 tokens yields a zero output.
* INT8 KV: symmetric, one fp32 scale per (token, KV head), separately for K and V;
  ``s = absmax / 127`` and ``q = clamp(round_half_even(x / s), -127, 127)``, both in
  IEEE fp32; ``absmax = 0`` gives ``s = 0`` and ``q = 0``.

Arithmetic is float64 throughout (inputs are converted exactly), except the INT8
quantiser, which the pages define on the stored fp32 values.
"""

from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# Paging arithmetic -- "分页注意力" section of "大模型工程（五）：推理优化核心技法"
# (chenk.top): KV is allocated in fixed-size blocks (16 tokens by default); a
# request of n tokens holds ceil(n / block_size) blocks and only its last block is
# partly filled.
# ---------------------------------------------------------------------------

def num_blocks_for(num_tokens: int, block_size: int) -> int:
    """Blocks a request of ``num_tokens`` tokens occupies (the page's 47 -> 3, 200 -> 13)."""
    if num_tokens < 0 or block_size <= 0:
        raise ValueError("num_tokens must be >= 0 and block_size > 0")
    return -(-num_tokens // block_size)


def kv_cache_bytes(batch: int, seq_len: int, num_layers: int, num_heads: int,
                   head_dim: int, dtype_bytes: int) -> int:
    """KV-cache size from section 2.1 of the gsyq.cn page:
    2 (K and V) x batch x seq_len x layers x heads x head_dim x bytes per element."""
    return 2 * batch * seq_len * num_layers * num_heads * head_dim * dtype_bytes


# ---------------------------------------------------------------------------
# Append -- "块管理器：分页如何运作" (block manager) of the chenk.top page: a growing
# request writes its new token into the slot its block table maps it to.
# ---------------------------------------------------------------------------

def append_scatter(k, v, k_cache, v_cache, slot_mapping, block_size):
    """Literal scatter of new tokens into the paged caches; returns new arrays.

    ``k``, ``v``: [T, Hkv, D]; caches: [NB, Hkv, bs, D]; ``slot_mapping``: [T] ints.
    Token ``t`` with ``slot >= 0`` lands at ``cache[slot // bs, :, slot % bs, :]``.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    for t in range(len(slot_mapping)):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        for h in range(k.shape[1]):
            k_out[blk, h, off, :] = k[t, h, :]
            v_out[blk, h, off, :] = v[t, h, :]
    return k_out, v_out


# ---------------------------------------------------------------------------
# INT8 KV quantiser -- "INT8 仅权重量化" of the chenk.top page gives the form
# w_q = round(w / s); "KV 缓存量化" of the same page and section 2.3 of the gsyq.cn
# page put one scale on each token (and head), never one global scale.
# ---------------------------------------------------------------------------

def quantize_rows_int8(x):
    """Symmetric per-row INT8 quantisation in IEEE fp32.

    ``x``: [..., D] values (converted to float32; bf16 inputs convert exactly).
    Returns ``(q int8 [..., D], s float32 [...])`` with ``s = absmax / 127`` and
    ``q = clamp(rint(x / s), -127, 127)`` (numpy's rint rounds half to even).
    """
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    q = np.zeros(x32.shape, dtype=np.int8)
    nz = s > 0
    if np.any(nz):
        ratio = (x32[nz] / s[nz][..., None]).astype(np.float32)
        q[nz] = np.clip(np.rint(ratio), -127, 127).astype(np.int8)
    return q, s


def dequantize_rows_int8(q, s):
    """Real value of stored INT8 codes: ``q * s`` evaluated in float64."""
    return np.asarray(q, dtype=np.float64) * np.asarray(s, dtype=np.float64)[..., None]


def append_scatter_int8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, block_size):
    """Quantise each new token's K and V rows per KV head, then scatter codes and scales.

    Caches: int8 [NB, Hkv, bs, D]; scales: float32 [NB, Hkv, bs]. Returns new arrays.
    """
    kq, ks = quantize_rows_int8(k)
    vq, vs = quantize_rows_int8(v)
    outs = [np.array(a, copy=True) for a in (k_cache, v_cache, k_scale, v_scale)]
    kc, vc, ksc, vsc = outs
    for t in range(len(slot_mapping)):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        for h in range(k.shape[1]):
            kc[blk, h, off, :] = kq[t, h, :]
            vc[blk, h, off, :] = vq[t, h, :]
            ksc[blk, h, off] = ks[t, h]
            vsc[blk, h, off] = vs[t, h]
    return kc, vc, ksc, vsc


# ---------------------------------------------------------------------------
# FP8 KV -- "FP8（及 H100/H200 硬件路径）" and "KV 缓存量化" of the chenk.top page:
# E4M3 (4 exponent, 3 mantissa bits) and E5M2 (5 exponent, 2 mantissa bits), the
# latter named for KV caches, with per-token scales computed online. The formats are
# taken as their usual definitions: E4M3 has exponent bias 7, no infinities, one NaN
# mantissa pattern (S.1111.111) and largest finite value 448; E5M2 has bias 15 and
# IEEE-style infinities/NaN, largest finite value 57344.
# ---------------------------------------------------------------------------

FP8_FORMATS = {"e4m3": (4, 3, 7), "e5m2": (5, 2, 15)}
FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def fp8_decode(codes, fmt):
    """Exact value (float64) of each FP8 byte code; NaN for NaN codes, +-inf for the
    E5M2 infinities."""
    e_bits, m_bits, bias = FP8_FORMATS[fmt]
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> m_bits) & ((1 << e_bits) - 1)
    m = c & ((1 << m_bits) - 1)
    frac = m / float(1 << m_bits)
    normal = (1.0 + frac) * np.power(2.0, e - bias)
    sub = frac * 2.0 ** (1 - bias)
    val = np.where(e == 0, sub, normal)
    if fmt == "e4m3":
        val = np.where((e == 15) & (m == 7), np.nan, val)
    else:
        val = np.where(e == 31, np.where(m == 0, np.inf, np.nan), val)
    return sign * val


def _fp8_finite_table(fmt):
    """(values ascending, codes) of every finite non-negative FP8 value."""
    codes = np.arange(0, 128)
    vals = fp8_decode(codes, fmt)
    keep = np.isfinite(vals)
    return vals[keep], codes[keep]


def fp8_round(x, fmt):
    """Round float32 values to the nearest FP8 code (ties to the even mantissa, i.e.
    the even code), saturating to the largest finite value; returns uint8 codes."""
    vals, codes = _fp8_finite_table(fmt)
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros(x.shape, dtype=np.uint8)
    flat_a, flat_out = a.reshape(-1), out.reshape(-1)
    neg = (x.reshape(-1) < 0)
    for i, v in enumerate(flat_a):
        if v >= vals[-1]:
            c = codes[-1]
        else:
            d = np.abs(vals - v)
            best = np.flatnonzero(d == d.min())
            c = codes[best[0]] if len(best) == 1 else codes[best[np.argmin(codes[best] % 2)]]
        flat_out[i] = (int(c) | (0x80 if neg[i] else 0)) if not (c == 0 and neg[i]) else 0x80
    return out


def quantize_rows_fp8(x, fmt):
    """Per-row FP8 quantisation in IEEE fp32: s = absmax / FP8_MAX, code =
    round_fp8(x / s); absmax = 0 gives s = 0 and zero codes. Returns (uint8 codes, s)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s = (amax / np.float32(FP8_MAX[fmt])).astype(np.float32)
    codes = np.zeros(x32.shape, dtype=np.uint8)
    nz = s > 0
    if np.any(nz):
        ratio = (x32[nz] / s[nz][..., None]).astype(np.float32)
        codes[nz] = fp8_round(ratio, fmt)
    return codes, s


def dequantize_rows_fp8(codes, s, fmt):
    return fp8_decode(codes, fmt) * np.asarray(s, dtype=np.float64)[..., None]


def append_scatter_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, block_size, fmt):
    """Quantise each new token's K and V rows per KV head to FP8, then scatter codes
    (uint8) and scales. Returns new arrays."""
    kq, ks = quantize_rows_fp8(k, fmt)
    vq, vs = quantize_rows_fp8(v, fmt)
    kc, vc, ksc, vsc = [np.array(a, copy=True) for a in (k_cache, v_cache, k_scale, v_scale)]
    for t in range(len(slot_mapping)):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        for h in range(k.shape[1]):
            kc[blk, h, off, :] = kq[t, h, :]
            vc[blk, h, off, :] = vq[t, h, :]
            ksc[blk, h, off] = ks[t, h]
            vsc[blk, h, off] = vs[t, h]
    return kc, vc, ksc, vsc


# ---------------------------------------------------------------------------
# Decode attention -- "两个特性截然不同的阶段" of the chenk.top page: one new query
# per request attends over that request's whole cached K/V; "分页注意力" of the same
# page: the cached tokens are reached through the request's block table.
# ---------------------------------------------------------------------------

def gather_sequence(cache, block_table_row, context_len, kv_head, block_size):
    """Contiguous [L, D] float64 copy of one sequence's cached rows for one KV head.

    Logical token ``t`` lives in physical block ``block_table_row[t // bs]`` at offset
    ``t % bs``; table entries past ``ceil(L / bs)`` are never read.
    """
    L = int(context_len)
    rows = []
    for t in range(L):
        phys = int(block_table_row[t // block_size])
        rows.append(np.asarray(cache[phys, kv_head, t % block_size, :], dtype=np.float64))
    if not rows:
        return np.zeros((0, cache.shape[-1]), dtype=np.float64)
    return np.stack(rows)


def attend_one_head(q, K, V, scale):
    """softmax(scale * K q) V for one head, float64, max-subtracted for stability.

    ``q``: [D]; ``K``, ``V``: [L, D]. Returns ([D] output, [L] weights). L = 0 gives a
    zero output and no weights. The dot products are elementwise sums (no BLAS), so
    the oracle runs on one core.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1], dtype=np.float64), np.zeros(0, dtype=np.float64)
    z = float(scale) * np.sum(K * q[None, :], axis=1)
    e = np.exp(z - np.max(z))
    w = e / np.sum(e)
    out = np.sum(w[:, None] * V, axis=0)
    return out, w


def _kv_head_of(h, group):
    return h // group


def decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, block_size=None):
    """Reference paged decode attention (MHA and GQA), float64.

    ``q``: [B, Hq, D]; caches: [NB, Hkv, bs, D] (real values, any float dtype);
    ``block_tables``: [B, MBS] ints; ``context_lens``: [B] ints. Returns [B, Hq, D]
    float64.
    """
    q = np.asarray(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    bs = int(block_size) if block_size is not None else k_cache.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    g = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for s in range(B):
        L = int(context_lens[s])
        for kvh in range(Hkv):
            K = gather_sequence(k_cache, block_tables[s], L, kvh, bs)
            V = gather_sequence(v_cache, block_tables[s], L, kvh, bs)
            for h in range(Hq):
                if _kv_head_of(h, g) != kvh:
                    continue
                out[s, h], _ = attend_one_head(q[s, h], K, V, scale)
    return out


def decode_attention_multi(q, k_cache, v_cache, block_tables, context_lens, scale,
                           block_size=None):
    """Paged attention for q_len new tokens per sequence at once (the verification pass
    of "推测解码" on the chenk.top page: the target model scores the k drafted tokens
    and the position after them, q_len = k + 1, in one pass), float64.

    ``q``: [B, q_len, Hq, D]. Every sequence's q_len newest tokens are already in the
    cache, so ``context_lens[s]`` counts them; new token i sits at position
    context_lens[s] - q_len + i and attends causally to positions 0 .. itself.
    Returns [B, q_len, Hq, D]. A sequence with context length 0 gets zeros.
    """
    q = np.asarray(q)
    B, n, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    bs = int(block_size) if block_size is not None else k_cache.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    g = Hq // Hkv
    out = np.zeros((B, n, Hq, D), dtype=np.float64)
    for s in range(B):
        L = int(context_lens[s])
        if L == 0:
            continue
        if L < n:
            raise ValueError("a sequence holds fewer tokens than its queries")
        for kvh in range(Hkv):
            K = gather_sequence(k_cache, block_tables[s], L, kvh, bs)
            V = gather_sequence(v_cache, block_tables[s], L, kvh, bs)
            for i in range(n):
                visible = L - n + i + 1            # positions 0 .. L - n + i
                for h in range(Hq):
                    if _kv_head_of(h, g) != kvh:
                        continue
                    out[s, i, h], _ = attend_one_head(q[s, i, h], K[:visible], V[:visible],
                                                      scale)
    return out


def gather_sequence_int8(codes, scales, block_table_row, context_len, kv_head, block_size):
    """Real [L, D] float64 values of one sequence's INT8 rows: code times its scale."""
    q = gather_sequence(codes, block_table_row, context_len, kv_head, block_size)
    L = int(context_len)
    s = np.array([float(scales[int(block_table_row[t // block_size]), kv_head, t % block_size])
                  for t in range(L)], dtype=np.float64)
    return q * s[:, None]


def decode_attention_int8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                          context_lens, scale, block_size=None):
    """Paged decode attention over an INT8 cache: the stored codes times their fp32
    per-(token, head) scales are the cached K/V values (exact in float64), then the
    same attention as :func:`decode_attention`.
    """
    q = np.asarray(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    bs = int(block_size) if block_size is not None else k_cache.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    g = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for s in range(B):
        L = int(context_lens[s])
        for kvh in range(Hkv):
            K = gather_sequence_int8(k_cache, k_scale, block_tables[s], L, kvh, bs)
            V = gather_sequence_int8(v_cache, v_scale, block_tables[s], L, kvh, bs)
            for h in range(Hq):
                if _kv_head_of(h, g) != kvh:
                    continue
                out[s, h], _ = attend_one_head(q[s, h], K, V, scale)
    return out


def gather_sequence_fp8(codes, scales, block_table_row, context_len, kv_head, block_size, fmt):
    """Real [L, D] float64 values of one sequence's FP8 rows: decoded code times scale."""
    c = gather_sequence(codes, block_table_row, context_len, kv_head, block_size)
    L = int(context_len)
    val = fp8_decode(c.astype(np.int64), fmt) if L else c
    s = np.array([float(scales[int(block_table_row[t // block_size]), kv_head, t % block_size])
                  for t in range(L)], dtype=np.float64)
    return val * s[:, None] if L else val


def decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                         scale, fmt, block_size=None):
    """Paged decode attention over an FP8 cache (codes decoded exactly, times their
    fp32 per-(token, head) scales), then the same attention as decode_attention."""
    q = np.asarray(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    bs = int(block_size) if block_size is not None else k_cache.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for s in range(B):
        L = int(context_lens[s])
        for kvh in range(Hkv):
            K = gather_sequence_fp8(k_cache, k_scale, block_tables[s], L, kvh, bs, fmt)
            V = gather_sequence_fp8(v_cache, v_scale, block_tables[s], L, kvh, bs, fmt)
            for h in range(Hq):
                if _kv_head_of(h, g) == kvh:
                    out[s, h], _ = attend_one_head(q[s, h], K, V, scale)
    return out


def decode_attention_multi_quantized(q, k_codes, v_codes, k_scale, v_scale, block_tables,
                                     context_lens, scale, fmt, block_size=None):
    """Multi-query paged attention (the causal rule of :func:`decode_attention_multi`)
    over a one-byte cache: ``fmt`` "int8", "e4m3" or "e5m2"; the cached K/V values are
    the codes (decoded exactly) times their fp32 per-(token, head) scales, the
    quantised caches of "KV 缓存量化" on the chenk.top page. float64, returns
    [B, q_len, Hq, D]."""
    q = np.asarray(q)
    B, n, Hq, D = q.shape
    Hkv = k_codes.shape[1]
    bs = int(block_size) if block_size is not None else k_codes.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    g = Hq // Hkv
    out = np.zeros((B, n, Hq, D), dtype=np.float64)
    for s in range(B):
        L = int(context_lens[s])
        if L == 0:
            continue
        if L < n:
            raise ValueError("a sequence holds fewer tokens than its queries")
        for kvh in range(Hkv):
            if fmt == "int8":
                K = gather_sequence_int8(k_codes, k_scale, block_tables[s], L, kvh, bs)
                V = gather_sequence_int8(v_codes, v_scale, block_tables[s], L, kvh, bs)
            else:
                K = gather_sequence_fp8(k_codes, k_scale, block_tables[s], L, kvh, bs, fmt)
                V = gather_sequence_fp8(v_codes, v_scale, block_tables[s], L, kvh, bs, fmt)
            for i in range(n):
                visible = L - n + i + 1            # positions 0 .. L - n + i
                for h in range(Hq):
                    if _kv_head_of(h, g) != kvh:
                        continue
                    out[s, i, h], _ = attend_one_head(q[s, i, h], K[:visible], V[:visible],
                                                      scale)
    return out


# ---------------------------------------------------------------------------
# Block moves -- "块管理器：分页如何运作" of the chenk.top page: a block shared under
# copy-on-write is copied to a fresh block before a request writes into it; under
# memory pressure a victim request's blocks are copied to pinned host memory and
# freed, and copied back into (new) blocks later.
# ---------------------------------------------------------------------------

def copy_blocks(cache, src_ids, dst_ids):
    """cache[dst_ids[i]] = cache[src_ids[i]] for every pair, all reads before any write.
    The pairs must not chain: no destination may also be a source or repeat."""
    src = [int(x) for x in src_ids]
    dst = [int(x) for x in dst_ids]
    if len(src) != len(dst):
        raise ValueError("src_ids and dst_ids differ in length")
    if len(set(dst)) != len(dst) or set(dst) & set(src):
        raise ValueError("copy pairs chain or repeat a destination")
    out = np.array(cache, copy=True)
    saved = [np.array(cache[b], copy=True) for b in src]
    for d, blk in zip(dst, saved):
        out[d] = blk
    return out


def swap_out_blocks(cache, block_ids):
    """The listed blocks stacked in list order: host[i] = cache[block_ids[i]]."""
    return np.stack([np.array(cache[int(b)], copy=True) for b in block_ids]) if len(block_ids) \
        else np.zeros((0,) + tuple(np.shape(cache)[1:]), dtype=np.asarray(cache).dtype)


def swap_in_blocks(cache, host, block_ids):
    """cache[block_ids[i]] = host[i]; the ids must be distinct. Returns a new array."""
    ids = [int(b) for b in block_ids]
    if len(set(ids)) != len(ids):
        raise ValueError("swap-in ids repeat")
    out = np.array(cache, copy=True)
    for i, b in enumerate(ids):
        out[b] = host[i]
    return out
