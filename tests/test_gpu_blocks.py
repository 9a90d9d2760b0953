"""GPU parity of whole-block moves against the oracle (bit-exact): the copy-on-write
block copy, eviction of blocks to pinned host memory and their return, for bf16 and
one-byte caches; bad ids are skipped and flagged; a fork followed by copy-on-write
appends leaves both requests' attention equal to the oracle's; a request swapped out
and back into other blocks decodes bit-identically."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_02_gb300.workloads import BlockAllocator, SequenceBlocks, make_workload
from parity_helpers import DECODE_ATOL

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_decode_02_gb300 import build_lib
    build_lib.build()
    import paged_kv_decode_02_gb300 as pk
    pk.load_library()
    return pk


def _np(t):
    t = t.detach().cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()


def _arrays(w):
    a = [w.k_cache, w.v_cache]
    if w.k_scale is not None:
        a += [w.k_scale, w.v_scale]
    return a


@pytest.mark.parametrize("name,kv", [("70b-gqa", None), ("int8", None), ("tiny", "fp8_e4m3")])
def test_copy_blocks_bit_exact(pk, name, kv):
    w = make_workload(name, device=DEV, num_seqs=4, kv_dtype=kv)
    rng = np.random.default_rng(1)
    perm = rng.permutation(w.num_blocks)
    n = min(24, w.num_blocks // 2)
    src, dst = perm[:n], perm[n:2 * n]
    before = [_np(t) for t in _arrays(w)]
    src_d = torch.tensor(src, dtype=torch.int32, device=DEV)
    dst_d = torch.tensor(dst, dtype=torch.int32, device=DEV)
    pk.copy_blocks(w.k_cache, w.v_cache, src_d, dst_d, w.k_scale, w.v_scale)
    torch.cuda.synchronize()
    for got, old in zip(_arrays(w), before):
        assert np.array_equal(_np(got), oracle.copy_blocks(old, src, dst))


def test_copy_blocks_skips_and_flags_bad_ids(pk):
    w = make_workload("tiny", device=DEV)
    before = [_np(t) for t in _arrays(w)]
    src = torch.tensor([3, 5, 7], dtype=torch.int32, device=DEV)
    dst = torch.tensor([9, w.num_blocks, 11], dtype=torch.int32, device=DEV)   # middle is bad
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk.copy_blocks(w.k_cache, w.v_cache, src, dst, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0x2
    for got, old in zip(_arrays(w), before):
        assert np.array_equal(_np(got), oracle.copy_blocks(old, [3, 7], [9, 11]))


@pytest.mark.parametrize("name,kv", [("70b-gqa", None), ("int8", None), ("tiny", "fp8_e5m2")])
def test_swap_out_and_in_bit_exact(pk, name, kv):
    w = make_workload(name, device=DEV, num_seqs=3, kv_dtype=kv)
    rng = np.random.default_rng(2)
    perm = rng.permutation(w.num_blocks)
    n = min(40, w.num_blocks // 2)
    out_ids, in_ids = perm[:n], perm[n:2 * n]
    arrays = _arrays(w)
    hosts = [torch.empty((n,) + tuple(t.shape[1:]), dtype=t.dtype).pin_memory() for t in arrays]
    while len(hosts) < 4:
        hosts.append(None)
    before = [_np(t) for t in arrays]
    ids = torch.tensor(out_ids, dtype=torch.int32, device=DEV)
    pk.swap_out(w.k_cache, w.v_cache, ids, hosts[0], hosts[1], w.k_scale, w.v_scale, hosts[2],
                hosts[3])
    torch.cuda.synchronize()
    for h, old in zip(hosts, before):
        assert np.array_equal(_np(h), oracle.swap_out_blocks(old, out_ids))
    ids_in = torch.tensor(in_ids, dtype=torch.int32, device=DEV)
    pk.swap_in(w.k_cache, w.v_cache, ids_in, hosts[0], hosts[1], w.k_scale, w.v_scale, hosts[2],
               hosts[3])
    torch.cuda.synchronize()
    for got, old, h in zip(arrays, before, hosts):
        assert np.array_equal(_np(got), oracle.swap_in_blocks(old, _np(h), in_ids))


def test_moves_check_buffers_before_launch(pk):
    """Host buffers too short for the listed blocks, caches that disagree and one-byte
    caches without their scales are refused by the binding; nothing launches."""
    lib = pk.pagedkv.load_library()
    w = make_workload("tiny", device=DEV)
    i8 = make_workload("tiny", device=DEV, kv_dtype="int8")
    ids = torch.tensor([1, 5, 9], dtype=torch.int32, device=DEV)
    short = torch.empty((2,) + tuple(w.k_cache.shape[1:]), dtype=torch.bfloat16).pin_memory()
    full = torch.empty((3,) + tuple(w.k_cache.shape[1:]), dtype=torch.bfloat16).pin_memory()
    n0 = lib.pkv_kernel_launch_count()
    with pytest.raises(ValueError):
        pk.swap_out(w.k_cache, w.v_cache, ids, short, full)
    with pytest.raises(ValueError):
        pk.swap_in(w.k_cache, w.v_cache, ids, full, short)
    with pytest.raises(ValueError):
        pk.copy_blocks(w.k_cache, w.v_cache[:-1], ids, ids + 1)
    with pytest.raises(TypeError):
        pk.copy_blocks(i8.k_cache, i8.v_cache, ids, ids + 1)                    # no scales
    hk = torch.empty((3,) + tuple(i8.k_cache.shape[1:]), dtype=torch.int8).pin_memory()
    hs = torch.empty((2,) + tuple(i8.k_scale.shape[1:]), dtype=torch.float32).pin_memory()
    with pytest.raises(ValueError):
        pk.swap_out(i8.k_cache, i8.v_cache, ids, hk, hk.clone().pin_memory(), i8.k_scale,
                    i8.v_scale, hs, hs.clone().pin_memory())                   # short scales
    assert lib.pkv_kernel_launch_count() == n0


def test_swap_refuses_pageable_host_memory(pk):
    from paged_kv_decode_02_gb300 import pagedkv
    w = make_workload("tiny", device=DEV)
    lib = pagedkv.load_library()
    host = torch.empty((2,) + tuple(w.k_cache.shape[1:]), dtype=torch.bfloat16)   # pageable
    ids = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    dims = pagedkv.Dims(0, w.num_kv_heads, w.num_kv_heads, w.head_dim, w.block_size,
                        w.num_blocks, 1)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.pkv_swap_out(p(host), p(host), None, None, p(w.k_cache), p(w.v_cache), None, None,
                          p(ids), 2, pagedkv.KV_BF16, ctypes.byref(dims), None, None)
    assert st == pagedkv.Status.ERR_HOST_MEMORY


def test_swap_round_trip_decodes_bit_identically(pk):
    """Evict three requests, let the pool hand their blocks to others, bring them back
    into fresh blocks with rewritten tables: the decode output is unchanged."""
    w = make_workload("70b-gqa", device=DEV, num_seqs=8, seed=31)
    ref = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w.scale)
    L = w.context_lens.cpu().numpy()
    tables = w.block_tables.cpu().numpy().copy()
    victims = [1, 4, 6]
    nblk = {s: -(-int(L[s]) // w.block_size) for s in victims}
    ids = np.concatenate([tables[s, :nblk[s]] for s in victims])
    host_k = torch.empty((len(ids),) + tuple(w.k_cache.shape[1:]), dtype=torch.bfloat16).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    pk.swap_out(w.k_cache, w.v_cache, torch.tensor(ids, dtype=torch.int32, device=DEV),
                host_k, host_v)
    # the freed blocks are overwritten (another request's data) ...
    ids_d = torch.tensor(ids, dtype=torch.int64, device=DEV)
    w.k_cache[ids_d] = float("nan")
    w.v_cache[ids_d] = float("nan")
    # ... and the victims come back into free blocks of the pool, in another order
    used = set(int(tables[s, j]) for s in range(w.num_seqs) if s not in victims
               for j in range(-(-int(L[s]) // w.block_size)))
    free = np.array(sorted(set(range(w.num_blocks)) - used), dtype=np.int64)
    new_ids = np.random.default_rng(3).permutation(free)[:len(ids)]
    assert len(new_ids) == len(ids) and not np.array_equal(new_ids, ids)
    pk.swap_in(w.k_cache, w.v_cache, torch.tensor(new_ids, dtype=torch.int32, device=DEV),
               host_k, host_v)
    off = 0
    for s in victims:
        tables[s, :nblk[s]] = new_ids[off:off + nblk[s]]
        off += nblk[s]
    out = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache,
                                    torch.from_numpy(tables).to(DEV), w.context_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_fork_copy_on_write_then_decode(pk):
    """Request b forks request a mid-block, then both append 5 tokens: a's first write
    into the shared last block moves a to a private copy (b then owns the original
    alone and writes in place); both decode as the oracle says."""
    bs, Hkv, Hq, D = 16, 2, 8, 128
    nb = 32
    alloc = BlockAllocator(nb, np.random.default_rng(4))
    gen = torch.Generator(device=DEV).manual_seed(5)
    k_cache = torch.randn((nb, Hkv, bs, D), generator=gen, device=DEV).to(torch.bfloat16)
    v_cache = torch.randn((nb, Hkv, bs, D), generator=gen, device=DEV).to(torch.bfloat16)
    a = SequenceBlocks(alloc, bs)
    slots = a.append_tokens(37)                    # 2 full blocks + 5 tokens
    toks = torch.randn((37, Hkv, D), generator=gen, device=DEV).to(torch.bfloat16)
    toks_v = torch.randn((37, Hkv, D), generator=gen, device=DEV).to(torch.bfloat16)
    pk.paged_kv_append(toks, toks_v, k_cache, v_cache,
                       torch.tensor(slots, dtype=torch.int64, device=DEV))
    b = SequenceBlocks(alloc, bs)
    b.fork_all(a)
    copies = []
    slots_a = a.append_tokens(5, copies)           # a writes first: a moves to the copy
    slots_b = b.append_tokens(5, copies)           # b is then the only owner: no copy
    assert len(copies) == 1
    src, dst = zip(*copies)
    pk.copy_blocks(k_cache, v_cache, torch.tensor(src, dtype=torch.int32, device=DEV),
                   torch.tensor(dst, dtype=torch.int32, device=DEV))
    new_k = torch.randn((10, Hkv, D), generator=gen, device=DEV).to(torch.bfloat16)
    new_v = torch.randn((10, Hkv, D), generator=gen, device=DEV).to(torch.bfloat16)
    pk.paged_kv_append(new_k, new_v, k_cache, v_cache,
                       torch.tensor(slots_a + slots_b, dtype=torch.int64, device=DEV))
    mbs = max(len(a.blocks), len(b.blocks))
    tables = torch.tensor([a.blocks + [nb + 7] * (mbs - len(a.blocks)),
                           b.blocks + [nb + 7] * (mbs - len(b.blocks))],
                          dtype=torch.int32, device=DEV)
    lens = torch.tensor([42, 42], dtype=torch.int32, device=DEV)
    q = torch.randn((2, Hq, D), generator=gen, device=DEV).to(torch.bfloat16)
    out = pk.paged_decode_attention(q, k_cache, v_cache, tables, lens, D ** -0.5)
    torch.cuda.synchronize()
    kc = k_cache.double().cpu().numpy()
    vc = v_cache.double().cpu().numpy()
    ref = oracle.decode_attention(q.double().cpu().numpy(), kc, vc, tables.cpu().numpy(),
                                  [42, 42], D ** -0.5)
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref))) <= DECODE_ATOL
    # each request reads its own 5 new tokens after the shared 37
    for s, lo in ((0, 0), (1, 5)):
        blocks = (a if s == 0 else b).blocks
        for t in range(5):
            pos = 37 + t
            row = k_cache[blocks[pos // bs], :, pos % bs]
            assert torch.equal(row, new_k[lo + t])
