"""GPU parity: the CUDA library against the fp64 CPU oracle on seeded inputs.

* append (bf16 scatter, INT8 and FP8 quantise + scatter): bit-exact;
* decode (bf16, INT8 and FP8 caches): max |gpu - oracle| <= 1e-2 on the bf16 output, on
  whole outputs at sizes the oracle finishes in seconds (several tiles, ragged tails,
  every group-size path) and on sampled outputs at the full workload sizes, in the
  launch configuration the benchmark uses.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_02_gb300.workloads import make_workload
from parity_helpers import (DECODE_ATOL, max_err, oracle_outputs, oracle_outputs_all,
                            sample_pairs, to_f64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_decode_02_gb300 import build_lib
    build_lib.build()
    import paged_kv_decode_02_gb300 as pk
    pk.load_library()
    return pk


def _decode(pk, w, **kw):
    if w.kv_dtype.startswith("fp8_"):
        return pk.paged_decode_attention_fp8(w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                             w.block_tables, w.context_lens, w.scale,
                                             fmt=w.kv_dtype[4:], **kw)
    if w.kv_dtype == "int8":
        return pk.paged_decode_attention_int8(w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                              w.block_tables, w.context_lens, w.scale, **kw)
    return pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                     w.scale, **kw)


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,kw", [("tiny", {}), ("70b-gqa", dict(num_seqs=5, head_dim=128)),
                                     ("7b", dict(num_seqs=3, lengths=[1, 17, 2048]))])
def test_append_bf16_bit_exact(pk, name, kw):
    w = make_workload(name, device=DEV, **kw)
    slots = w.slot_mapping.clone()
    slots[0] = -1                                   # a skipped token
    kc0, vc0 = w.k_cache.clone(), w.v_cache.clone()
    pk.paged_kv_append(w.new_k, w.new_v, w.k_cache, w.v_cache, slots)
    torch.cuda.synchronize()
    ref_k, ref_v = oracle.append_scatter(
        w.new_k.view(torch.int16).cpu().numpy(), w.new_v.view(torch.int16).cpu().numpy(),
        kc0.view(torch.int16).cpu().numpy(), vc0.view(torch.int16).cpu().numpy(),
        slots.cpu().numpy(), w.block_size)
    assert np.array_equal(w.k_cache.view(torch.int16).cpu().numpy(), ref_k)
    assert np.array_equal(w.v_cache.view(torch.int16).cpu().numpy(), ref_v)


@pytest.mark.parametrize("D,bs", [(128, 32), (128, 16), (64, 16)])
def test_append_int8_bit_exact(pk, D, bs):
    w = make_workload("int8", device=DEV, num_seqs=6, lengths=[1, 31, 32, 33, 100, 64],
                      head_dim=D, block_size=bs)
    gen = torch.Generator(device=DEV).manual_seed(7)
    k = (torch.randn(w.new_k.shape, generator=gen, device=DEV) *
         torch.logspace(-3, 3, w.new_k.shape[0], device=DEV)[:, None, None]).to(torch.bfloat16)
    v = torch.randn(w.new_v.shape, generator=gen, device=DEV).to(torch.bfloat16)
    v[1] = 0                                         # an all-zero row -> scale 0, codes 0
    k[2, 0, :4] = torch.tensor([127.0, 2.5, -2.5, 3.5])  # exact halves at unit scale
    k[2, 0, 4:] = 0
    slots = w.slot_mapping.clone()
    slots[3] = -1
    before = [t.clone() for t in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    pk.paged_kv_append_int8(k, v, w.k_cache, w.v_cache, w.k_scale, w.v_scale, slots)
    torch.cuda.synchronize()
    ref = oracle.append_scatter_int8(k.float().cpu().numpy(), v.float().cpu().numpy(),
                                     *[t.cpu().numpy() for t in before], slots.cpu().numpy(), bs)
    got = [t.cpu().numpy() for t in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    for a, b in zip(got, ref):
        assert np.array_equal(a.view(np.uint8) if a.dtype == np.int8 else a.view(np.uint32),
                              b.view(np.uint8) if b.dtype == np.int8 else b.view(np.uint32))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("D,bs", [(128, 32), (64, 16)])
def test_append_fp8_bit_exact(pk, fmt, D, bs):
    w = make_workload("fp8-" + fmt, device=DEV, num_seqs=6, lengths=[1, 31, 32, 33, 100, 64],
                      head_dim=D, block_size=bs)
    gen = torch.Generator(device=DEV).manual_seed(9)
    # magnitudes over six decades, so that small entries of a row land on subnormal
    # codes or round to (signed) zero
    k = (torch.randn(w.new_k.shape, generator=gen, device=DEV) *
         torch.logspace(-3, 3, w.new_k.shape[0], device=DEV)[:, None, None]).to(torch.bfloat16)
    v = (torch.randn(w.new_v.shape, generator=gen, device=DEV) *
         torch.logspace(-4, 0, D, device=DEV)).to(torch.bfloat16)
    v[1] = 0                                         # an all-zero row -> scale 0, codes 0
    slots = w.slot_mapping.clone()
    slots[3] = -1
    before = [t.clone() for t in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    pk.paged_kv_append_fp8(k, v, w.k_cache, w.v_cache, w.k_scale, w.v_scale, slots, fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.append_scatter_fp8(k.float().cpu().numpy(), v.float().cpu().numpy(),
                                    *[t.cpu().numpy() for t in before], slots.cpu().numpy(), bs,
                                    fmt)
    got = [t.cpu().numpy() for t in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    for a, b in zip(got, ref):
        assert np.array_equal(a.view(np.uint8) if a.dtype == np.uint8 else a.view(np.uint32),
                              b.view(np.uint8) if b.dtype == np.uint8 else b.view(np.uint32))


# ---------------------------------------------------------------------------
# decode, whole outputs at small sizes
# ---------------------------------------------------------------------------

def test_decode_tiny_with_poisoned_unused_slots(pk):
    w = make_workload("tiny", device=DEV, poison_unused=True)
    out = _decode(pk, w)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL


SHAPES = [
    # (name, Hq, Hkv, D, bs, lengths)
    ("mha-d128-bs16", 8, 8, 128, 16, [1, 15, 16, 17, 100, 333]),
    ("mha-d64-bs32", 4, 4, 64, 32, [64, 3, 95, 200]),
    ("g2-d128-bs32", 8, 4, 128, 32, [33, 7, 250]),
    ("g3-d64-bs16", 6, 2, 64, 16, [48, 49, 1, 130]),
    ("g4-d128-bs16", 16, 4, 128, 16, [1, 16, 47, 200, 513]),
    ("g8-d128-bs16", 16, 2, 128, 16, [40, 700, 9, 64]),
    ("g8-d64-bs32", 16, 2, 64, 32, [31, 32, 33, 300]),
    ("g5-d128-bs32", 10, 2, 128, 32, [100, 5]),
    ("g16-d128-bs16", 32, 2, 128, 16, [77, 260]),
    ("g32-d64-bs16", 64, 2, 64, 16, [90, 17]),
]


KV_WORKLOAD = {"bf16": "70b-gqa", "int8": "int8", "fp8_e4m3": "fp8-e4m3",
               "fp8_e5m2": "fp8-e5m2"}


@pytest.mark.parametrize("kv", list(KV_WORKLOAD))
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_decode_small_shapes(pk, shape, kv):
    _, Hq, Hkv, D, bs, lengths = shape
    w = make_workload(KV_WORKLOAD[kv], device=DEV, num_q_heads=Hq, num_kv_heads=Hkv,
                      head_dim=D, block_size=bs, lengths=lengths, seed=11, poison_unused=True)
    out = _decode(pk, w)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL


def test_decode_empty_and_single_token_sequences(pk):
    w = make_workload("70b-gqa", device=DEV, num_q_heads=16, num_kv_heads=4, head_dim=128,
                      lengths=[0, 1, 0, 16, 1], seed=3)
    out = _decode(pk, w)
    torch.cuda.synchronize()
    got = to_f64(out)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL
    # one token: the output is that token's V row (rounded to bf16)
    blk = w.block_tables[1, 0].item()
    for h in range(16):
        np.testing.assert_array_equal(got[1, h], to_f64(w.v_cache[blk, h // 4, 0]))


def test_decode_single_long_sequence_split_many_ways(pk):
    """B = 1: one long context is cut across many workers and merged."""
    w = make_workload("70b-gqa", device=DEV, lengths=[20000], num_q_heads=8, num_kv_heads=1,
                      seed=5)
    out = _decode(pk, w)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8_e5m2"])
def test_decode_single_long_mha_sequence(pk, kv):
    """B = 1, one KV head: one 32K-token context over every worker (more partials than
    the merge stages at once)."""
    name = "7b" if kv == "bf16" else KV_WORKLOAD[kv]
    w = make_workload(name, device=DEV, lengths=[32768], num_q_heads=1, num_kv_heads=1,
                      seed=8)
    out = _decode(pk, w)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL


def test_decode_permuted_placement_is_bit_identical(pk):
    w = make_workload("70b-gqa", device=DEV, num_seqs=6, seed=9)
    out1 = _decode(pk, w).clone()
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(1)).to(DEV)
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt = w.block_tables.clone().long()
    valid = bt < w.num_blocks
    bt[valid] = perm[bt[valid]]
    w.k_cache, w.v_cache, w.block_tables = k2, v2, bt.to(torch.int32)
    out2 = _decode(pk, w)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_decode_status_flags_bad_tables(pk):
    w = make_workload("70b-gqa", device=DEV, num_seqs=4, num_q_heads=16, num_kv_heads=4, seed=4)
    w.block_tables[1, 0] = w.num_blocks + 100        # out-of-range block id
    w.context_lens[2] = w.block_tables.shape[1] * w.block_size + 5  # longer than its table
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _decode(pk, w, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & 0x2 and st & 0x1 and not st & 0x4
    got = to_f64(out)
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    good = [(s, h) for s in (0, 3) for h in range(16)]
    w.context_lens[2] = 1   # keep the oracle away from the invalid rows
    ref = oracle_outputs(w, good)
    assert max_err(out, ref, good) <= DECODE_ATOL


def test_decode_reuses_caller_workspace_and_output(pk):
    w = make_workload("70b-gqa", device=DEV, num_seqs=8, seed=6)
    need = pk.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     w.block_size, w.num_blocks, w.max_blocks_per_seq)
    ws = torch.zeros(need + (1 << 20), dtype=torch.uint8, device=DEV)
    out = torch.full_like(w.q, float("nan"))
    r1 = _decode(pk, w, out=out, workspace=ws).clone()
    r2 = _decode(pk, w, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(r1, r2)
    ref = oracle_outputs(w)
    assert max_err(r2, ref) <= DECODE_ATOL
    # the same workspace, never re-zeroed, serves other shapes in between
    for other in (make_workload("7b", device=DEV, lengths=[3000, 5, 700], seed=2),
                  make_workload("70b-gqa", device=DEV, lengths=[20000], num_q_heads=16,
                                num_kv_heads=1, seed=3)):
        o2 = _decode(pk, other, workspace=ws)
        torch.cuda.synchronize()
        assert max_err(o2, oracle_outputs(other)) <= DECODE_ATOL
    r3 = _decode(pk, w, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(r1, r3)


def test_binding_checks_buffers_before_launch(pk):
    """The binding refuses, before anything launches, a workspace or status word the
    kernels could not use (host memory, wrong dtype) and tensors whose shapes disagree
    with the caches (output, new rows, slots, scales); it counts a caller workspace of
    any dtype in bytes."""
    lib = pk.pagedkv.load_library()
    w = make_workload("70b-gqa", device=DEV, num_seqs=4, seed=8)
    need = pk.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     w.block_size, w.num_blocks, w.max_blocks_per_seq)
    ref = _decode(pk, w)
    torch.cuda.synchronize()
    n0 = lib.pkv_kernel_launch_count()
    with pytest.raises(ValueError):
        _decode(pk, w, workspace=torch.zeros(need, dtype=torch.uint8))           # host memory
    with pytest.raises(TypeError):
        _decode(pk, w, status=torch.zeros(1, dtype=torch.int64, device=DEV))
    with pytest.raises(ValueError):
        _decode(pk, w, status=torch.zeros(1, dtype=torch.int32))                 # host memory
    # shapes the kernels would address past a buffer's end
    with pytest.raises(ValueError):
        _decode(pk, w, out=torch.empty_like(w.q)[:-1])                          # short out
    with pytest.raises(ValueError):
        pk.paged_kv_append(w.new_k, w.new_v, w.k_cache, w.v_cache, w.slot_mapping[:-1])
    with pytest.raises(ValueError):
        pk.paged_kv_append(w.new_k[..., :64].contiguous(), w.new_v, w.k_cache, w.v_cache,
                           w.slot_mapping)                                     # wrong head_dim
    i8 = make_workload("int8", device=DEV, num_seqs=2, lengths=[40, 9], block_size=16)
    with pytest.raises(ValueError):
        pk.paged_decode_attention_int8(i8.q, i8.k_cache, i8.v_cache, i8.k_scale[:-1],
                                       i8.v_scale, i8.block_tables, i8.context_lens, i8.scale)
    with pytest.raises(ValueError):
        pk.paged_kv_append_int8(i8.new_k, i8.new_v, i8.k_cache, i8.v_cache, i8.k_scale,
                                i8.v_scale[:-1], i8.slot_mapping)
    assert lib.pkv_kernel_launch_count() == n0
    # a float32 workspace holding the bytes is used as it is (its size counted in bytes)
    ws = torch.zeros(-(-need // 4) + 64, dtype=torch.float32, device=DEV)
    out = _decode(pk, w, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_kernel_launch_counts_per_call(pk):
    """The library's launch counter (what bench.py reports as gpu_launches) against the
    kernels each call is documented to launch."""
    lib = pk.pagedkv.load_library()

    def launches(fn):
        torch.cuda.synchronize()
        n0 = lib.pkv_kernel_launch_count()
        fn()
        torch.cuda.synchronize()
        return lib.pkv_kernel_launch_count() - n0

    mha = make_workload("7b", device=DEV, lengths=[700, 30, 2048], seed=7)
    gqa = make_workload("70b-gqa", device=DEV, num_seqs=6, seed=8)
    spec = make_workload("spec-70b", device=DEV, num_q_heads=16, num_kv_heads=2, q_len=6,
                         lengths=[600, 6, 130], seed=9)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert launches(lambda: pk.paged_kv_append(mha.new_k, mha.new_v, mha.k_cache, mha.v_cache,
                                               mha.slot_mapping)) == 1
    # MHA, head_dim 128, bf16, no status word: cut units folded inside the decode kernel
    assert launches(lambda: _decode(pk, mha)) == 1
    assert launches(lambda: _decode(pk, mha, status=status)) == 2      # + validating merge
    assert launches(lambda: _decode(pk, gqa)) == 2                     # decode + merge
    # tcgen05 multi-query kernel: cut heads folded at the CTA tail
    assert launches(lambda: pk.paged_decode_attention_multi(
        spec.q, spec.k_cache, spec.v_cache, spec.block_tables, spec.context_lens,
        spec.scale)) == 1
    assert launches(lambda: pk.paged_decode_attention_multi(
        spec.q, spec.k_cache, spec.v_cache, spec.block_tables, spec.context_lens, spec.scale,
        status=status)) == 2
    assert int(status.item()) == 0


# ---------------------------------------------------------------------------
# decode at the full workload sizes, sampled outputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["7b", "70b-gqa", "prefix", "int8", "int8-bs16", "fp8-e5m2",
                                  "fp8-e4m3"])
def test_decode_full_size_sampled(pk, name):
    w = make_workload(name, device=DEV)
    if w.kv_dtype == "bf16":
        pk.paged_kv_append(w.new_k, w.new_v, w.k_cache, w.v_cache, w.slot_mapping)
    elif w.kv_dtype.startswith("fp8_"):
        pk.paged_kv_append_fp8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                               w.slot_mapping, fmt=w.kv_dtype[4:])
    else:
        pk.paged_kv_append_int8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                w.slot_mapping)
    out = _decode(pk, w)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    pairs = sample_pairs(w, 24)
    ref = oracle_outputs(w, pairs)
    assert max_err(out, ref, pairs) <= DECODE_ATOL


@pytest.mark.parametrize("name", ["70b-gqa", "7b", "prefix", "int8", "int8-bs16", "fp8-e5m2",
                                  "fp8-e4m3"])
def test_decode_full_size_whole_output(pk, name):
    """Every output row of a full-size workload, after the step's append, against the
    oracle (run on all host cores): 70b-gqa has cut units everywhere (470 of its 512
    (sequence, KV head) units are split over several workers and merged), 7b folds its
    parts inside the kernel, prefix reads its shared blocks from every table, the one-byte
    workloads quantise their new tokens on append."""
    w = make_workload(name, device=DEV)
    if w.kv_dtype == "bf16":
        pk.paged_kv_append(w.new_k, w.new_v, w.k_cache, w.v_cache, w.slot_mapping)
    elif w.kv_dtype.startswith("fp8_"):
        pk.paged_kv_append_fp8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                               w.slot_mapping, fmt=w.kv_dtype[4:])
    else:
        pk.paged_kv_append_int8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                w.slot_mapping)
    out = _decode(pk, w)
    torch.cuda.synchronize()
    ref = oracle_outputs_all(w)
    assert max_err(out, ref) <= DECODE_ATOL


# ---------------------------------------------------------------------------
# cascade decode for a prefix shared by the whole batch
# ---------------------------------------------------------------------------

def _cascade(pk, w, prefix_blocks, **kw):
    return pk.paged_decode_attention_cascade(w.q, w.k_cache, w.v_cache, w.block_tables,
                                             w.context_lens, prefix_blocks, w.scale, **kw)


CASCADE_SHAPES = [
    # (Hq, Hkv, D, bs, prefix tokens, suffix lengths)
    (32, 8, 128, 16, 160, [16, 1, 33, 0, 200, 7]),
    (16, 16, 128, 16, 64, [5, 100, 0]),
    (8, 2, 64, 32, 96, [40, 3, 64, 1, 500]),
    (64, 4, 128, 32, 32, [10, 70]),
    (12, 4, 64, 16, 48, [0, 0, 9]),
]


@pytest.mark.parametrize("shape", CASCADE_SHAPES, ids=[f"c{i}" for i in range(len(CASCADE_SHAPES))])
def test_cascade_small_shapes(pk, shape):
    Hq, Hkv, D, bs, pre, suf = shape
    lengths = [pre + x for x in suf]
    w = make_workload("prefix", device=DEV, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                      block_size=bs, lengths=lengths, prefix_tokens=pre, seed=13,
                      poison_unused=True)
    out = _cascade(pk, w, pre // bs)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL
    plain = _decode(pk, w)
    torch.cuda.synchronize()
    assert float((out.float() - plain.float()).abs().max()) <= DECODE_ATOL


def test_cascade_row_tiles_and_ragged_prefix_tail(pk):
    # 70 sequences x 4 query heads per KV head = 280 query rows (two full 128-row tiles
    # and a ragged one); a 21-block prefix ends 5 blocks into its third 128-token tile
    rng = np.random.default_rng(5)
    pre, bs = 21 * 16, 16
    lengths = [pre + int(x) for x in rng.integers(0, 100, size=70)]
    w = make_workload("prefix", device=DEV, num_q_heads=16, num_kv_heads=4, head_dim=128,
                      block_size=bs, lengths=lengths, prefix_tokens=pre, seed=21,
                      poison_unused=True)
    out = _cascade(pk, w, pre // bs)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL


def test_cascade_scores_growing_across_prefix_tiles(pk):
    # Prefix keys scaled by 1, 5, 9, 13 in successive 128-token tiles: each tile's
    # maximum score exceeds the previous tiles' by far more than 2^8, so the prefix
    # kernel's accumulated output must be rescaled between tiles. 700 x 1 query rows
    # per KV head keep the grid above one wave, hence one prefix split on any GPU.
    # Such peaked weights make each output nearly one V row, so V is scaled by 1/4
    # (exact in bf16) to keep outputs in the range the bf16 tolerance is set for.
    pre, bs = 512, 16
    rng = np.random.default_rng(6)
    lengths = [pre + int(x) for x in rng.integers(0, 17, size=700)]
    w = make_workload("prefix", device=DEV, num_q_heads=32, num_kv_heads=32, head_dim=128,
                      block_size=bs, lengths=lengths, prefix_tokens=pre, seed=22)
    kc = w.k_cache.clone()
    for j in range(pre // bs):
        phys = int(w.block_tables[0, j])
        kc[phys] = (kc[phys].float() * (1 + 4 * (j * bs // 128))).to(torch.bfloat16)
    w.k_cache = kc
    w.v_cache = w.v_cache * 0.25
    out = _cascade(pk, w, pre // bs)
    torch.cuda.synchronize()
    pairs = sample_pairs(w, 48, seed=3)
    ref = oracle_outputs(w, pairs)
    assert max_err(out, ref, pairs) <= DECODE_ATOL
    plain = _decode(pk, w)
    torch.cuda.synchronize()
    assert float((out.float() - plain.float()).abs().max()) <= DECODE_ATOL


@pytest.mark.parametrize("scale", [0.0, -0.125], ids=["zero", "negative"])
def test_cascade_zero_and_negative_scale(pk, scale):
    # scale 0 weighs every position equally; a negative scale flips the ordering of
    # the scores (the prefix ends 3 blocks into its second 128-token tile)
    pre, bs = 11 * 16, 16
    w = make_workload("prefix", device=DEV, num_q_heads=16, num_kv_heads=4, head_dim=64,
                      block_size=bs, lengths=[pre + x for x in (0, 5, 40, 17, 90)],
                      prefix_tokens=pre, seed=23, poison_unused=True)
    w.scale = scale
    out = _cascade(pk, w, pre // bs)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL


@pytest.mark.parametrize("B,bs", [(128, 16), (256, 32)], ids=["4x16", "8x32"])
def test_cascade_four_and_eight_row_tiles(pk, B, bs):
    # 4 query heads per KV head: 128 sequences make 4 row tiles of 128 query rows per KV
    # head, 256 sequences 8 row tiles over blocks of 32 (4 blocks per 128-token tile)
    pre = 160 if bs == 16 else 192
    rng = np.random.default_rng(B + bs)
    lengths = [pre + int(x) for x in rng.integers(0, 41, size=B)]
    w = make_workload("prefix", device=DEV, num_q_heads=16, num_kv_heads=4, head_dim=128,
                      block_size=bs, lengths=lengths, prefix_tokens=pre, seed=24,
                      poison_unused=True)
    out = _cascade(pk, w, pre // bs)
    torch.cuda.synchronize()
    pairs = sample_pairs(w, 40, seed=5)
    ref = oracle_outputs(w, pairs)
    assert max_err(out, ref, pairs) <= DECODE_ATOL


def test_cascade_full_prefix_workload(pk):
    """The benchmark's headline step (append, then the cascade decode of the full prefix
    workload), every output row against the oracle run on all host cores."""
    w = make_workload("prefix", device=DEV)
    pk.paged_kv_append(w.new_k, w.new_v, w.k_cache, w.v_cache, w.slot_mapping)
    out = _cascade(pk, w, 2048 // w.block_size)
    torch.cuda.synchronize()
    ref = oracle_outputs_all(w)
    assert max_err(out, ref) <= DECODE_ATOL


def _cascade_q8(pk, w, prefix_blocks, **kw):
    return pk.paged_decode_attention_cascade_q8(
        w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale, w.block_tables, w.context_lens,
        prefix_blocks, w.scale, fmt=w.kv_dtype[4:] if w.kv_dtype != "int8" else "e5m2", **kw)


CASCADE_Q8 = [
    # (id, B, Hq, Hkv, D, bs, prefix tokens, suffix lengths)
    ("g4-bs16", 6, 16, 4, 128, 16, 256, [0, 5, 16, 17, 100, 300]),
    ("g8-bs32-d64", 5, 16, 2, 64, 32, 320, [1, 31, 64, 200, 0]),
    ("g1-bs16", 4, 4, 4, 128, 16, 144, [7, 0, 60, 129]),
]


@pytest.mark.parametrize("kvt", ["int8", "fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("case", CASCADE_Q8, ids=[c[0] for c in CASCADE_Q8])
def test_cascade_q8_small_shapes(pk, case, kvt):
    """Shared-prefix decode over one-byte caches: whole outputs against the oracle, with
    and without a status word (the latter validates the tables)."""
    _, B, Hq, Hkv, D, bs, pre, suf = case
    w = make_workload("prefix", device=DEV, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                      block_size=bs, lengths=[pre + x for x in suf], prefix_tokens=pre,
                      kv_dtype=kvt, seed=41, poison_unused=True)
    out = _cascade_q8(pk, w, pre // bs)
    torch.cuda.synchronize()
    ref = oracle_outputs(w)
    assert max_err(out, ref) <= DECODE_ATOL
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out2 = _cascade_q8(pk, w, pre // bs, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert max_err(out2, ref) <= DECODE_ATOL


@pytest.mark.parametrize("kvt", ["int8", "fp8_e5m2"])
def test_cascade_q8_full_prefix_workload(pk, kvt):
    """The prefix workload over a one-byte cache: quantise-append the step's tokens, then
    the cascade decode; every output row against the oracle (all host cores)."""
    w = make_workload("prefix", device=DEV, kv_dtype=kvt)
    if kvt == "int8":
        pk.paged_kv_append_int8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                w.slot_mapping)
    else:
        pk.paged_kv_append_fp8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                               w.slot_mapping, fmt=kvt[4:])
    out = _cascade_q8(pk, w, 2048 // w.block_size)
    torch.cuda.synchronize()
    ref = oracle_outputs_all(w)
    assert max_err(out, ref) <= DECODE_ATOL


def test_cascade_flags_a_table_without_the_prefix(pk):
    pre, bs = 64, 16
    w = make_workload("prefix", device=DEV, num_q_heads=16, num_kv_heads=4, head_dim=128,
                      lengths=[pre + 20, pre + 5, pre + 40], prefix_tokens=pre, seed=14)
    bt = w.block_tables.clone()
    bt[1, 2] = (w.block_tables[1, 2] + 1) % w.num_blocks     # no longer the shared block
    w.block_tables = bt
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _cascade(pk, w, pre // bs, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x8
    got = to_f64(out)
    assert np.all(got[1] == 0)
    good = [(s, h) for s in (0, 2) for h in range(16)]
    ref = oracle_outputs(w, good)
    assert max_err(out, ref, good) <= DECODE_ATOL
