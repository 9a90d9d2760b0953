"""Pins for the oracle's block moves (copy-on-write copy, swap-out gather, swap-in
scatter; "块管理器：分页如何运作" of the chenk.top page) and the host allocator's
copy-on-write and eviction bookkeeping.

The moves are checked through what must hold around them: a copied block equals its
source bit for bit and nothing else changes; swapping a request out and back into
different blocks leaves its attention output bit-identical (against the pinned
decode oracle); after a fork, writes by one request never show in the other's
attention, and each sees exactly its own tokens. Planted mistakes must fail.
"""

import numpy as np
import pytest

import oracle
from oracle import paged_attention as pa
from paged_kv_decode_02_gb300.workloads import BlockAllocator, SequenceBlocks

BS, HKV, D = 4, 2, 3


def _cache(nb, seed):
    return np.random.default_rng(seed).standard_normal((nb, HKV, BS, D))


def test_copy_blocks_copies_exactly_the_pairs():
    c = _cache(8, 0)
    out = oracle.copy_blocks(c, [1, 5], [6, 2])
    assert np.array_equal(out[6], c[1]) and np.array_equal(out[2], c[5])
    for b in (0, 1, 3, 4, 5, 7):
        assert np.array_equal(out[b], c[b])
    assert np.array_equal(oracle.copy_blocks(c, [], []), c)


def test_copy_blocks_refuses_chained_pairs():
    c = _cache(4, 1)
    with pytest.raises(ValueError):
        oracle.copy_blocks(c, [0, 1], [1, 2])          # 1 is read and written
    with pytest.raises(ValueError):
        oracle.copy_blocks(c, [0, 1], [3, 3])          # 3 written twice


def test_swap_round_trip_into_new_blocks_keeps_attention():
    rng = np.random.default_rng(2)
    alloc = BlockAllocator(12, rng)
    a, b = SequenceBlocks(alloc, BS), SequenceBlocks(alloc, BS)
    a.append_tokens(10)
    b.append_tokens(7)
    k, v = _cache(12, 3), _cache(12, 4)
    q = rng.standard_normal((1, HKV * 2, D))
    before = oracle.decode_attention(q, k, v, np.array([a.blocks]), [10], 0.6)
    n = len(a.blocks)
    old = a.swap_out()
    hk, hv = oracle.swap_out_blocks(k, old), oracle.swap_out_blocks(v, old)
    assert hk.shape == (n, HKV, BS, D) and np.array_equal(hk[1], k[old[1]])
    b.append_tokens(9)                              # the pool moves on meanwhile
    new = a.swap_in(n)
    k2, v2 = oracle.swap_in_blocks(k, hk, new), oracle.swap_in_blocks(v, hv, new)
    after = oracle.decode_attention(q, k2, v2, np.array([new]), [10], 0.6)
    assert np.array_equal(before, after)


def test_fork_then_write_is_copy_on_write():
    rng = np.random.default_rng(5)
    alloc = BlockAllocator(10, rng)
    a = SequenceBlocks(alloc, BS)
    slots_a = a.append_tokens(6)                    # blocks [x full, y with 2 tokens]
    k = np.zeros((10, HKV, BS, D))
    v = np.zeros((10, HKV, BS, D))
    toks_k = rng.standard_normal((6, HKV, D))
    toks_v = rng.standard_normal((6, HKV, D))
    k, v = oracle.append_scatter(toks_k, toks_v, k, v, slots_a, BS)
    b = SequenceBlocks(alloc, BS)
    b.fork_all(a)
    assert alloc.refcount[a.blocks[1]] == 2
    copies = []
    slots_b = b.append_tokens(3, copies)            # b writes into the shared block
    assert len(copies) == 1 and copies[0][0] == a.blocks[1] and b.blocks[1] == copies[0][1]
    assert alloc.refcount[a.blocks[1]] == 1 and b.blocks[0] == a.blocks[0]
    src, dst = zip(*copies)
    k, v = oracle.copy_blocks(k, src, dst), oracle.copy_blocks(v, src, dst)
    new_k, new_v = rng.standard_normal((3, HKV, D)), rng.standard_normal((3, HKV, D))
    k, v = oracle.append_scatter(new_k, new_v, k, v, slots_b, BS)
    q = rng.standard_normal((1, HKV, D))
    # a still sees exactly its 6 tokens
    out_a = oracle.decode_attention(q, k, v, np.array([a.blocks]), [6], 0.8)
    priv_a = oracle.decode_attention(q, _blocks_of(toks_k), _blocks_of(toks_v),
                                     np.array([[0, 1]]), [6], 0.8)
    assert np.array_equal(out_a, priv_a)
    # b sees a's 6 tokens followed by its own 3
    kb, vb = np.concatenate([toks_k, new_k]), np.concatenate([toks_v, new_v])
    out_b = oracle.decode_attention(q, k, v, np.array([b.blocks]), [9], 0.8)
    priv_b = oracle.decode_attention(q, _blocks_of(kb), _blocks_of(vb), np.array([[0, 1, 2]]),
                                     [9], 0.8)
    assert np.array_equal(out_b, priv_b)


def _blocks_of(tokens):
    """[T, HKV, D] rows laid out as private blocks 0, 1, ... ([nb, HKV, BS, D])."""
    T = tokens.shape[0]
    nb = -(-T // BS)
    out = np.zeros((nb, HKV, BS, D))
    for t in range(T):
        out[t // BS, :, t % BS] = tokens[t]
    return out


def test_write_into_shared_block_without_copy_list_is_refused():
    alloc = BlockAllocator(4)
    a = SequenceBlocks(alloc, BS)
    a.append_tokens(2)
    b = SequenceBlocks(alloc, BS)
    b.fork_all(a)
    with pytest.raises(ValueError):
        b.append_tokens(1)


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _fails(fn, *args):
    try:
        fn(*args)
    except Exception:
        return True
    return False


def test_pins_catch_copy_in_the_wrong_direction(monkeypatch):
    orig = pa.copy_blocks
    for mod in (pa, oracle):
        monkeypatch.setattr(mod, "copy_blocks", lambda c, s, d: orig(c, d, s))
    assert _fails(test_copy_blocks_copies_exactly_the_pairs)
    assert _fails(test_fork_then_write_is_copy_on_write)


def test_pins_catch_swap_out_in_reverse_order(monkeypatch):
    orig = pa.swap_out_blocks
    for mod in (pa, oracle):
        monkeypatch.setattr(mod, "swap_out_blocks", lambda c, ids: orig(c, list(ids)[::-1]))
    assert _fails(test_swap_round_trip_into_new_blocks_keeps_attention)
