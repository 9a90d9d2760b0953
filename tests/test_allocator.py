"""Host block allocator: the block-manager behaviour of "大模型工程（五）：推理优化核心技法"
(chenk.top), section "块管理器：分页如何运作" -- free list, grow by appending a block,
refcounted sharing under copy-on-write (fork adds, free drops, release at zero)."""

import numpy as np
import pytest

from paged_kv_decode_02_gb300.workloads import (BlockAllocator, SequenceBlocks, build_tables,
                                                make_workload)


def test_grow_appends_a_block_every_block_size_tokens():
    alloc = BlockAllocator(8, np.random.default_rng(0))
    sb = SequenceBlocks(alloc, 16)
    slots = sb.append_tokens(47)
    assert len(sb.blocks) == 3 and alloc.num_free == 5
    assert slots[0] == sb.blocks[0] * 16 and slots[16] == sb.blocks[1] * 16
    assert slots[-1] == sb.blocks[2] * 16 + 14
    sb.append_tokens(1)          # 48th token fills block 3 exactly
    assert len(sb.blocks) == 3
    sb.append_tokens(1)          # 49th opens a fourth block
    assert len(sb.blocks) == 4


def test_fork_and_free_refcounts():
    alloc = BlockAllocator(4)
    a = SequenceBlocks(alloc, 16)
    a.append_tokens(32)
    b = SequenceBlocks(alloc, 16)
    b.fork_prefix(a, 32)
    assert all(alloc.refcount[x] == 2 for x in a.blocks)
    a.release()
    assert alloc.num_free == 2                       # still held by b
    assert all(alloc.refcount[x] == 1 for x in b.blocks)
    b.release()
    assert alloc.num_free == 4 and np.all(alloc.refcount == 0)
    with pytest.raises(ValueError):
        alloc.free(0)


def test_pool_exhaustion_raises():
    alloc = BlockAllocator(2)
    sb = SequenceBlocks(alloc, 16)
    sb.append_tokens(32)
    with pytest.raises(MemoryError):
        sb.append_tokens(1)


def test_prefix_tables_share_blocks_with_refcount_batch():
    rng = np.random.default_rng(1)
    lengths = 2048 + rng.integers(16, 513, size=6)
    tables, last, NB, alloc = build_tables(lengths, 16, rng, shared_prefix_tokens=2048)
    pre = tables[0, :128]
    for s in range(6):
        assert np.array_equal(tables[s, :128], pre)
        n = -(-int(lengths[s]) // 16)
        assert np.all(tables[s, n:] >= NB)          # poison past the request's blocks
        assert last[s] // 16 == tables[s, n - 1]     # last token lands in the private tail
    assert np.all(alloc.refcount[pre] == 6)
    private = np.concatenate([tables[s, 128:-(-int(lengths[s]) // 16)] for s in range(6)])
    assert len(set(private.tolist())) == len(private)
    assert not set(private.tolist()) & set(pre.tolist())


def test_named_workloads_shapes():
    w = make_workload("tiny")
    assert w.q.shape == (4, 8, 64) and w.k_cache.shape == (64, 8, 16, 64)
    assert w.block_tables.shape[0] == 4
    assert int(w.context_lens.min()) >= 1 and int(w.context_lens.max()) <= 64
    w = make_workload("70b-gqa", num_seqs=8, head_dim=64)
    L = w.context_lens.numpy()
    assert L.min() >= 128 and L.max() <= 32768
    w = make_workload("int8", num_seqs=2, lengths=[40, 3])
    assert w.k_cache.dtype.is_floating_point is False and w.k_scale.shape[-1] == 32
