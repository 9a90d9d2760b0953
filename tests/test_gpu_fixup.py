"""GPU parity of the in-kernel stream-K fixup (single-token decode with one query head
per KV head, bf16 cache, head_dim 128, no status word): units cut between decode warps
are folded by the warp that completes them, through counters in the workspace that
carry a launch tag instead of being cleared.

Checked against the fp64 oracle: dense cuts (more blocks than warps) and sparse cuts
(fewer blocks than warps: every block of a unit is its own part), a workspace that
starts as garbage, repeated calls on one workspace, and replays of a CUDA graph whose
query changes between replays.
"""

import numpy as np
import pytest
import torch

from paged_kv_decode_02_gb300.workloads import make_workload
from parity_helpers import DECODE_ATOL, max_err, oracle_outputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pk():
    from paged_kv_decode_02_gb300 import build_lib
    build_lib.build()
    import paged_kv_decode_02_gb300 as pk
    pk.load_library()
    return pk


def _workspace(pk, w, fill):
    n = pk.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                  w.block_size, w.num_blocks, w.block_tables.shape[1])
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=DEV)
    if fill == "ones":
        ws.fill_(0xFF)
    else:
        gen = torch.Generator(device=DEV).manual_seed(11)
        ws.copy_(torch.randint(0, 256, ws.shape, generator=gen, device=DEV, dtype=torch.int32)
                 .to(torch.uint8))
    return ws


# dense: 32 heads x (128 + 3 + 63 + 33) blocks, more than the decode warps;
# sparse: 32 heads x (7 + 3 + 1) blocks, fewer than the warps (a part per block)
CASES = {
    "dense-bs16": dict(num_seqs=4, lengths=[2048, 37, 1000, 513]),
    "dense-bs32": dict(num_seqs=4, lengths=[2048, 37, 1000, 513], block_size=32),
    "sparse": dict(num_seqs=3, lengths=[100, 33, 16]),
    "with-empty": dict(num_seqs=4, lengths=[700, 0, 1, 300]),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("fill", ["ones", "random"])
def test_fixup_garbage_workspace_and_repeats(pk, case, fill):
    w = make_workload("7b", device=DEV, **CASES[case])
    ref = oracle_outputs(w)
    ws = _workspace(pk, w, fill)
    out = torch.empty_like(w.q)
    for _ in range(3):  # the counters each call leaves behind serve the next
        out.fill_(float("nan"))
        pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                  w.scale, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert max_err(out, ref) <= DECODE_ATOL


@pytest.mark.parametrize("case", ["dense-bs16", "sparse"])
def test_fixup_graph_replays(pk, case):
    w = make_workload("7b", device=DEV, **CASES[case])
    ws = _workspace(pk, w, "random")
    out = torch.empty_like(w.q)
    q = w.q.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm-up outside the capture
        pk.paged_decode_attention(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                  w.scale, out=out, workspace=ws)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pk.paged_decode_attention(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                  w.scale, out=out, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(5)
    for _ in range(4):
        q.copy_(torch.randn(q.shape, generator=gen, device=DEV).to(q.dtype))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        w.q = q.clone()
        assert max_err(out, oracle_outputs(w)) <= DECODE_ATOL
