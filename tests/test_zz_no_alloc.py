"""pkv_decode_bf16_noalloc: decode for callers that cannot allocate device memory.

Some callers of this library have no allocator to hand it a workspace -- code that
runs inside another runtime's memory pool, plugins that may not call cudaMalloc, or
latency-critical paths where no allocation may happen. The no-allocation entry point
serves them from a fixed scratch array kept in the library's device image. This test
calls it through the C ABI, twice in a row on different shapes (so the second call
finds the first call's leftovers in the shared scratch), and checks each result
against the ordinary entry point given a freshly allocated workspace, within the
tolerance the other decode tests use. A third call passes a device status word, which
sends the split-KV parts through the merge kernel (it reads the partials the decode
left in the shared scratch): the status must stay 0 and the result must match too. It
also checks that shapes beyond the fixed limits are refused without a launch.

The file name sorts last so that a run stopping at the first failure has already run
every other test; it builds and loads the library itself so that it also passes alone.
"""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DECODE_ATOL = 1e-2
NOALLOC_SCRATCH_BYTES = 16 << 20  # PKV_NOALLOC_SCRATCH_BYTES in include/pagedkv.h
NOALLOC_MAX_SEQ_HEADS = 65536     # PKV_NOALLOC_MAX_SEQ_HEADS in include/pagedkv.h
# the first PKV_NOALLOC_MAX_SEQ_HEADS 8-byte words of the scratch hold counters only
NOALLOC_MAX_BYTES = NOALLOC_SCRATCH_BYTES - 8 * NOALLOC_MAX_SEQ_HEADS


def _lib():
    from paged_kv_decode_02_gb300 import build_lib, pagedkv
    build_lib.build()
    return pagedkv, pagedkv.load_library()


def _args(w, pagedkv):
    dims = pagedkv.Dims(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                        w.num_blocks, w.max_blocks_per_seq)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return dims, p


def _reference(lib, pagedkv, w, stream):
    dims, p = _args(w, pagedkv)
    need = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(dims), pagedkv.KV_BF16,
                                          ctypes.byref(need)) == 0
    ws = torch.zeros(int(need.value), dtype=torch.uint8, device="cuda")  # zeroed before first use
    out = torch.empty_like(w.q)
    st = lib.pkv_decode_bf16(p(out), p(w.q), p(w.k_cache), p(w.v_cache), p(w.block_tables),
                             p(w.context_lens), w.scale, ctypes.byref(dims), p(ws), ws.numel(),
                             None, stream)
    assert st == 0
    return out, int(need.value)


def test_noalloc_decode_matches_allocating_entry_point():
    from paged_kv_decode_02_gb300.workloads import make_workload
    pagedkv, lib = _lib()
    torch.cuda.set_device(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [
        make_workload("70b-gqa", device="cuda", num_seqs=12, seed=21),           # g = 8
        make_workload("7b", device="cuda", lengths=[3, 2048, 700, 1, 64], seed=22),  # MHA
    ]
    # (workload, pass a status word): the third call repeats the MHA shape, whose
    # 2048-token sequence is split over several workers, with a status word
    for w, with_status in ((cases[0], False), (cases[1], False), (cases[1], True)):
        ref, need = _reference(lib, pagedkv, w, stream)
        assert need <= NOALLOC_MAX_BYTES
        dims, p = _args(w, pagedkv)
        out = torch.full_like(w.q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda") if with_status else None
        st = lib.pkv_decode_bf16_noalloc(p(out), p(w.q), p(w.k_cache), p(w.v_cache),
                                         p(w.block_tables), p(w.context_lens), w.scale,
                                         ctypes.byref(dims),
                                         p(status) if with_status else None, stream)
        assert st == 0, lib.pkv_status_string(st)
        torch.cuda.synchronize()
        if with_status:
            assert int(status.item()) == 0
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - ref.double().cpu().numpy()))) <= DECODE_ATOL


def test_noalloc_refuses_shapes_beyond_its_scratch():
    pagedkv, lib = _lib()
    torch.cuda.set_device(0)
    # 64 query heads on 2 KV heads needs ~20 MB of partials, more than the fixed 16 MiB
    dims = pagedkv.Dims(8, 64, 2, 128, 16, 1024, 64)
    need = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(dims), pagedkv.KV_BF16,
                                          ctypes.byref(need)) == 0
    assert need.value > NOALLOC_MAX_BYTES
    p = ctypes.c_void_p(256)
    st = lib.pkv_decode_bf16_noalloc(p, p, p, p, p, p, 0.1, ctypes.byref(dims), None, None)
    assert st == pagedkv.Status.ERR_WORKSPACE


def test_noalloc_refuses_more_sequence_heads_than_its_counters():
    pagedkv, lib = _lib()
    torch.cuda.set_device(0)
    # 2100 sequences x 32 KV heads = 67200 (sequence, KV head) counters, over the limit,
    # on a shape whose workspace alone would fit
    dims = pagedkv.Dims(2100, 32, 32, 64, 16, 4096, 4)
    need = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(dims), pagedkv.KV_BF16,
                                          ctypes.byref(need)) == 0
    assert need.value <= NOALLOC_MAX_BYTES
    assert 2100 * 32 > NOALLOC_MAX_SEQ_HEADS
    p = ctypes.c_void_p(256)
    st = lib.pkv_decode_bf16_noalloc(p, p, p, p, p, p, 0.1, ctypes.byref(dims), None, None)
    assert st == pagedkv.Status.ERR_WORKSPACE
