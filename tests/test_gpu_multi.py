"""GPU parity of multi-query paged decode (q_len new tokens per sequence, causal; the
verification pass of speculative decoding) against the fp64 oracle: whole outputs
at small sizes covering every group size, ragged lengths, contexts made only of the
new tokens and long contexts cut between many workers; sampled outputs at the full
spec-70b size after appending the step's tokens; status flags."""

import numpy as np
import pytest
import torch

from paged_kv_decode_02_gb300.workloads import make_workload
from parity_helpers import (DECODE_ATOL, oracle_outputs_all, oracle_outputs_multi,
                            oracle_outputs_multi_q8, to_f64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_decode_02_gb300 import build_lib
    build_lib.build()
    import paged_kv_decode_02_gb300 as pk
    pk.load_library()
    return pk


def _run(pk, w, **kw):
    return pk.paged_decode_attention_multi(w.q, w.k_cache, w.v_cache, w.block_tables,
                                           w.context_lens, w.scale, **kw)


def _err(out, ref, triples=None):
    got = to_f64(out)
    if triples is None:
        assert np.all(np.isfinite(got))
        return float(np.max(np.abs(got - ref)))
    return float(max(np.max(np.abs(got[s, i, h] - ref[s, i, h])) for (s, i, h) in triples))


SHAPES = [
    # (id, Hq, Hkv, D, bs, q_len, lengths)
    ("mha-q2", 4, 4, 128, 16, 2, [2, 17, 100, 0, 33]),
    ("mha-q6-d64-bs32", 4, 4, 64, 32, 6, [6, 7, 64, 65, 300]),
    ("g2-q3", 8, 4, 128, 16, 3, [3, 16, 19, 250]),
    ("g4-q4", 16, 4, 128, 16, 4, [4, 5, 31, 200, 513]),
    ("g8-q6", 16, 2, 128, 16, 6, [6, 40, 700, 12, 0, 64]),
    ("g8-q16-bs32", 16, 2, 128, 32, 16, [16, 17, 300, 1000]),
    ("g16-q2-d64", 32, 2, 64, 16, 2, [90, 17, 2]),
    ("g5-q5", 10, 2, 128, 32, 5, [100, 5, 37]),
    # 48..128 rows per KV head take the tcgen05 kernel, more than 128 the wide mma.sync one
    ("g16-q4-d64", 32, 2, 64, 16, 4, [4, 5, 129, 300, 0, 77]),
    ("g8-q8-bs32", 16, 2, 128, 32, 8, [8, 9, 130, 600]),
    ("g16-q8", 32, 2, 128, 16, 8, [8, 200, 1500, 127, 129]),
    ("g16-q12-d64", 32, 2, 64, 16, 12, [12, 40, 150]),
    # tcgen05 with groups whose rows do not form whole 8-row atoms (plain row stores)
    ("g12-q4", 24, 2, 128, 16, 4, [4, 60, 300, 129]),
    ("g4-q16-d64-bs32", 8, 2, 64, 32, 16, [16, 40, 500]),
    # more than 64 rows over bf16 with D 128: two softmax warps per lane quarter, each
    # storing its half of a row (plain row stores for g 6, TMA boxes of 32 rows for g 32)
    ("g6-q16-pair", 12, 2, 128, 16, 16, [16, 40, 700, 129, 0]),
    ("g32-q3-pair", 64, 2, 128, 16, 3, [3, 50, 400]),
]

# chunks of chunked prefill: more than 128 rows per KV head, run as equal tcgen05 row
# tiles (the last one padded when the tiles do not divide the rows), with ragged causal
# tails and contexts that hold only the chunk
CHUNKS = [
    # (id, Hq, Hkv, D, bs, q_len, lengths)
    ("g8-q64", 16, 2, 128, 16, 64, [64, 65, 300, 1000, 0, 127]),
    ("g8-q256", 16, 2, 128, 16, 256, [256, 300, 1300]),
    ("g4-q256-d64-bs32", 8, 2, 64, 32, 256, [256, 513, 900]),
    ("g6-q100", 12, 2, 128, 16, 100, [100, 101, 450]),       # g 6: plain row stores
    ("g1-q131-bs32", 2, 2, 128, 32, 131, [131, 200, 0]),     # 2 tiles of 66, the last padded
    ("g8-q17", 16, 2, 64, 16, 17, [17, 50, 333]),            # 2 tiles of 68 rows
]


@pytest.mark.parametrize("shape", CHUNKS, ids=[s[0] for s in CHUNKS])
def test_multi_prefill_chunks(pk, shape):
    _, Hq, Hkv, D, bs, n, lengths = shape
    w = make_workload("spec-70b", device=DEV, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                      block_size=bs, lengths=lengths, q_len=n, seed=31, poison_unused=True)
    out = _run(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_all(w)) <= DECODE_ATOL
    # the same call with a status word (the split-KV merge kernel folds the cut units)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out2 = _run(pk, w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert _err(out2, oracle_outputs_all(w)) <= DECODE_ATOL


def test_multi_prefill_chunk_full_size(pk):
    """A 256-token chunk for each of 16 requests with the 70b-gqa length mix (2048 query
    rows per KV head, 16 row tiles), after appending the chunk: every output row."""
    w = make_workload("chunk-70b", device=DEV)
    pk.paged_kv_append(w.new_k, w.new_v, w.k_cache, w.v_cache, w.slot_mapping)
    out = _run(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_all(w)) <= DECODE_ATOL


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_multi_small_shapes(pk, shape):
    _, Hq, Hkv, D, bs, n, lengths = shape
    w = make_workload("spec-70b", device=DEV, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                      block_size=bs, lengths=lengths, q_len=n, seed=13, poison_unused=True)
    out = _run(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_multi(w)) <= DECODE_ATOL


@pytest.mark.parametrize("Hq,Hkv,n", [(8, 1, 4), (1, 1, 8)])
def test_multi_long_context_split_many_ways(pk, Hq, Hkv, n):
    """One long context over every worker: the segments holding only the last block
    leave fully masked rows for the early query tokens, which the merge must skip."""
    w = make_workload("spec-70b", device=DEV, lengths=[20000], num_q_heads=Hq,
                      num_kv_heads=Hkv, q_len=n, seed=14)
    out = _run(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_multi(w)) <= DECODE_ATOL


@pytest.mark.parametrize("Hq,Hkv,n", [(16, 2, 6), (16, 2, 16), (32, 2, 4)],
                         ids=["48rows-split", "128rows", "64rows-split"])
def test_tc_scores_growing_across_tiles(pk, Hq, Hkv, n):
    """Keys scaled by 1, 5, 9, ... in successive 128-token tiles of every sequence: each
    tile's maximum score exceeds the previous tiles' by far more than 2^8, so the tcgen05
    kernel rescales O and the row sums between tiles (with split rows when a KV head has
    at most 64 rows, and across the MMAs it issues as their inputs become ready). V is
    scaled by 1/4 (exact in bf16) to keep the peaked outputs in the range the bf16
    tolerance is set for."""
    lengths = [700, 1000, 390, 129]
    w = make_workload("spec-70b", device=DEV, num_q_heads=Hq, num_kv_heads=Hkv, q_len=n,
                      lengths=lengths, seed=41)
    kc = w.k_cache.clone()
    bs = w.block_size
    for s_, L in enumerate(lengths):
        for j in range((L + bs - 1) // bs):
            phys = int(w.block_tables[s_, j])
            kc[phys] = (kc[phys].float() * (1 + 4 * (j * bs // 128))).to(torch.bfloat16)
    w.k_cache = kc
    w.v_cache = w.v_cache * 0.25
    out = _run(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_multi(w)) <= DECODE_ATOL


def test_multi_single_token_matches_decode(pk):
    w = make_workload("70b-gqa", device=DEV, num_seqs=6, seed=15)
    a = pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                  w.scale)
    b = pk.paged_decode_attention_multi(w.q[:, None], w.k_cache, w.v_cache, w.block_tables,
                                        w.context_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b[:, 0])


@pytest.mark.parametrize("name", ["spec-70b", "spec-70b-q16"])
def test_multi_full_size_after_append(pk, name):
    """The spec-70b steps (6 and 16 new tokens per request): append them, then verify;
    every output row against the oracle (all host cores)."""
    w = make_workload(name, device=DEV)
    pk.paged_kv_append(w.new_k, w.new_v, w.k_cache, w.v_cache, w.slot_mapping)
    out = _run(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_all(w)) <= DECODE_ATOL


def test_multi_full_size_128_rows(pk):
    """spec-70b lengths with 16 new tokens per request: 128 query rows per KV head."""
    w = make_workload("spec-70b", device=DEV, q_len=16)
    out = _run(pk, w)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    L = w.context_lens.cpu().numpy()
    triples = {(int(np.argmax(L)), 0, 0), (int(np.argmax(L)), 15, w.num_q_heads - 1),
               (int(np.argmin(L)), 15, 7)}
    while len(triples) < 24:
        triples.add((int(rng.integers(w.num_seqs)), int(rng.integers(w.q_len)),
                     int(rng.integers(w.num_q_heads))))
    triples = sorted(triples)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    assert _err(out, oracle_outputs_multi(w, triples), triples) <= DECODE_ATOL


def test_multi_flags_context_shorter_than_queries(pk):
    w = make_workload("spec-70b", device=DEV, num_q_heads=16, num_kv_heads=2,
                      lengths=[40, 9, 0], q_len=4, seed=16)
    lens = w.context_lens.clone()
    lens[1] = 2                               # 0 < L < q_len
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pk.paged_decode_attention_multi(w.q, w.k_cache, w.v_cache, w.block_tables, lens,
                                          w.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1
    got = to_f64(out)
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    ref = oracle_outputs_multi(w)
    assert float(np.max(np.abs(got[0] - ref[0]))) <= DECODE_ATOL


def test_multi_rejects_bad_query_length(pk):
    w = make_workload("spec-70b", device=DEV, num_seqs=2, q_len=2, lengths=[5, 9])
    # one more new token than PKV_MAX_QUERY_LEN (256)
    q = torch.zeros((2, 257, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(pk.PagedKVError):
        pk.paged_decode_attention_multi(q, w.k_cache, w.v_cache, w.block_tables,
                                        w.context_lens, w.scale)


# tcgen05 kernel (q_len * g query rows per KV head in 48..128): a head of 157 tiles cut
# over most CTAs, an empty sequence, fewer tiles than CTAs; two-token windows (new
# token 0 of a 9-token context) where the bf16 weights must be normalised by their own
# sum to stay inside the tolerance
TC_CASES = {
    "tc-64rows-long": dict(num_q_heads=16, num_kv_heads=2, q_len=8, lengths=[20000, 9, 300]),
    "tc-128rows-empty": dict(num_q_heads=16, num_kv_heads=2, q_len=16,
                             lengths=[3000, 0, 16, 1200]),
    "tc-48rows-sparse": dict(num_q_heads=16, num_kv_heads=2, q_len=6, lengths=[600, 6, 130]),
}


def _tc_workspace(pk, w, fill):
    n = pk.multi_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                 w.block_size, w.num_blocks, w.block_tables.shape[1], w.q_len)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=DEV)
    if fill == "ones":
        ws.fill_(0xFF)
    else:
        gen = torch.Generator(device=DEV).manual_seed(12)
        ws.copy_(torch.randint(0, 256, ws.shape, generator=gen, device=DEV, dtype=torch.int32)
                 .to(torch.uint8))
    return ws


@pytest.mark.parametrize("case", sorted(TC_CASES))
@pytest.mark.parametrize("fill", ["ones", "random"])
def test_tc_garbage_workspace_and_repeats(pk, case, fill):
    w = make_workload("spec-70b", device=DEV, seed=21, poison_unused=True, **TC_CASES[case])
    ref = oracle_outputs_multi(w)
    ws = _tc_workspace(pk, w, fill)
    out = torch.empty_like(w.q)
    for _ in range(3):  # one workspace for every call, never cleared
        out.fill_(float("nan"))
        _run(pk, w, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert _err(out, ref) <= DECODE_ATOL


def test_tc_graph_replays(pk):
    w = make_workload("spec-70b", device=DEV, seed=22, **TC_CASES["tc-64rows-long"])
    ws = _tc_workspace(pk, w, "random")
    out = torch.empty_like(w.q)
    q = w.q.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm-up outside the capture
        pk.paged_decode_attention_multi(q, w.k_cache, w.v_cache, w.block_tables,
                                        w.context_lens, w.scale, out=out, workspace=ws)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pk.paged_decode_attention_multi(q, w.k_cache, w.v_cache, w.block_tables,
                                        w.context_lens, w.scale, out=out, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(6)
    for _ in range(3):
        q.copy_(torch.randn(q.shape, generator=gen, device=DEV).to(q.dtype))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        w.q = q.clone()
        assert _err(out, oracle_outputs_multi(w)) <= DECODE_ATOL


# ---------------------------------------------------------------------------
# one-byte caches (INT8, FP8 E4M3 / E5M2 codes with per-(token, KV head) scales)
# ---------------------------------------------------------------------------

def _run_q8(pk, w, **kw):
    return pk.paged_decode_attention_multi_q8(w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                              w.block_tables, w.context_lens, w.scale,
                                              fmt=w.kv_dtype[4:] if w.kv_dtype != "int8"
                                              else "e5m2", **kw)


Q8_SHAPES = [
    # (id, Hq, Hkv, D, bs, q_len, lengths): 16, 48, 128 and several row tiles of rows
    ("g8-q2", 16, 2, 128, 16, 2, [2, 17, 300, 0, 129]),
    ("g8-q6-bs32", 16, 2, 128, 32, 6, [6, 40, 700, 33]),
    ("g8-q16-d64", 16, 2, 64, 16, 16, [16, 100, 1000]),
    ("g4-q64", 8, 2, 128, 16, 64, [64, 65, 500]),
    ("g1-q3-mha", 4, 4, 128, 32, 3, [3, 90, 257]),
]


@pytest.mark.parametrize("kvt", ["int8", "fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("shape", Q8_SHAPES, ids=[s[0] for s in Q8_SHAPES])
def test_multi_q8_small_shapes(pk, shape, kvt):
    _, Hq, Hkv, D, bs, n, lengths = shape
    w = make_workload("spec-70b", device=DEV, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                      block_size=bs, lengths=lengths, q_len=n, seed=33, kv_dtype=kvt,
                      poison_unused=True)
    out = _run_q8(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_multi_q8(w)) <= DECODE_ATOL
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out2 = _run_q8(pk, w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert _err(out2, oracle_outputs_multi_q8(w)) <= DECODE_ATOL


@pytest.mark.parametrize("kvt", ["int8", "fp8_e5m2"])
def test_multi_q8_full_size_after_append(pk, kvt):
    """The spec-70b step over a one-byte cache: quantise and append the 6 new tokens of
    every request, then verify; every output row against the oracle."""
    w = make_workload("spec-70b", device=DEV, kv_dtype=kvt)
    if kvt == "int8":
        pk.paged_kv_append_int8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                w.slot_mapping)
    else:
        pk.paged_kv_append_fp8(w.new_k, w.new_v, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                               w.slot_mapping, fmt=kvt[4:])
    out = _run_q8(pk, w)
    torch.cuda.synchronize()
    assert _err(out, oracle_outputs_all(w)) <= DECODE_ATOL


def test_multi_q8_single_token_is_decode(pk):
    w = make_workload("int8", device=DEV, num_seqs=4, lengths=[5, 300, 1000, 0], seed=34)
    a = pk.paged_decode_attention_int8(w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                       w.block_tables, w.context_lens, w.scale)
    b = pk.paged_decode_attention_multi_q8(w.q[:, None], w.k_cache, w.v_cache, w.k_scale,
                                           w.v_scale, w.block_tables, w.context_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b[:, 0])
