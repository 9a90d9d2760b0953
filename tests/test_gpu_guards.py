"""Guard bytes around the caller's buffers: every decode path writes its output and uses
its workspace strictly inside the bytes it was given.

The output and the workspace are views into larger device buffers whose head and tail
(4 KiB each, which keeps the views 256-byte aligned) hold a fill pattern; the workspace
view is exactly the size the library asks for. After the call both guards must still
hold the pattern, and the result must equal the same call on ordinary buffers. Paths:
single-token decode with the in-kernel fold (MHA bf16), with the merge kernel (GQA on
the tensor cores), INT8 and FP8 caches, multi-query decode on mma.sync and on tcgen05,
and the cascade.
"""

import pytest
import torch

from paged_kv_decode_02_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 4096
FILL = 0xA5


@pytest.fixture(scope="module")
def pk():
    from paged_kv_decode_02_gb300 import build_lib
    build_lib.build()
    import paged_kv_decode_02_gb300 as pk
    pk.load_library()
    return pk


def _guarded(nbytes):
    """(whole buffer, view of nbytes in its middle); the view starts GUARD bytes in."""
    buf = torch.full((GUARD + nbytes + GUARD,), FILL, dtype=torch.uint8, device=DEV)
    return buf, buf[GUARD:GUARD + nbytes]


def _guards_intact(buf, nbytes):
    return bool((buf[:GUARD] == FILL).all()) and bool((buf[GUARD + nbytes:] == FILL).all())


def _dims(w):
    return (w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
            w.num_blocks, w.max_blocks_per_seq)


def _single(pk, w, **kw):
    if w.kv_dtype == "int8":
        return pk.paged_decode_attention_int8(w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                              w.block_tables, w.context_lens, w.scale, **kw)
    if w.kv_dtype.startswith("fp8_"):
        return pk.paged_decode_attention_fp8(w.q, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                             w.block_tables, w.context_lens, w.scale,
                                             fmt=w.kv_dtype[4:], **kw)
    return pk.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                     w.context_lens, w.scale, **kw)


def _single_ws(pk, w):
    kv = {"bf16": pk.pagedkv.KV_BF16, "int8": pk.pagedkv.KV_INT8,
          "fp8_e4m3": pk.pagedkv.KV_FP8_E4M3, "fp8_e5m2": pk.pagedkv.KV_FP8_E5M2}[w.kv_dtype]
    return pk.decode_workspace_bytes(*_dims(w), kv_dtype=kv)


def _multi(pk, w, **kw):
    return pk.paged_decode_attention_multi(w.q, w.k_cache, w.v_cache, w.block_tables,
                                           w.context_lens, w.scale, **kw)


CASES = {
    # single-token decode, MHA bf16 head_dim 128: split parts folded inside the kernel
    "mha-fold": ("single", dict(name="7b", lengths=[3000, 5, 700, 0], seed=2)),
    # GQA group 8 on the tensor cores, block pairs, merge kernel
    "gqa-merge": ("single", dict(name="70b-gqa", num_seqs=8, seed=6)),
    "int8": ("single", dict(name="int8", lengths=[700, 33, 2000], seed=4)),
    "fp8-e4m3": ("single", dict(name="fp8-e4m3", lengths=[700, 33, 2000], seed=4)),
    # 16 query rows per KV head: mma.sync multi-query path
    "multi-mma": ("multi", dict(name="spec-70b", lengths=[900, 40, 3000], q_len=2, seed=7)),
    # 48 query rows per KV head: tcgen05 kernel
    "multi-tc": ("multi", dict(name="spec-70b", lengths=[900, 40, 3000], q_len=6, seed=7)),
    "cascade": ("cascade", dict(name="prefix", num_q_heads=32, num_kv_heads=8,
                                lengths=[160 + x for x in (16, 1, 33, 0, 200, 7)],
                                prefix_tokens=160, seed=13)),
}


@pytest.mark.parametrize("case", list(CASES))
def test_decode_stays_inside_output_and_workspace(pk, case):
    kind, kw = CASES[case]
    kw = dict(kw)
    w = make_workload(kw.pop("name"), device=DEV, **kw)
    if kind == "single":
        need = _single_ws(pk, w)
        call = lambda **a: _single(pk, w, **a)  # noqa: E731
    elif kind == "multi":
        need = pk.multi_workspace_bytes(*_dims(w), w.q.shape[1])
        call = lambda **a: _multi(pk, w, **a)  # noqa: E731
    else:
        pre = kw["prefix_tokens"] // w.block_size
        need = pk.cascade_workspace_bytes(*_dims(w), pre)
        call = lambda **a: pk.paged_decode_attention_cascade(  # noqa: E731
            w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, pre, w.scale, **a)
    ref = call()
    out_bytes = w.q.numel() * w.q.element_size()
    obuf, oview = _guarded(out_bytes)
    wbuf, wview = _guarded(need)
    out = oview.view(torch.bfloat16).view(w.q.shape)
    for _ in range(2):   # the second call finds the first one's leftovers in the workspace
        got = call(out=out, workspace=wview)
        torch.cuda.synchronize()
        assert got.data_ptr() == out.data_ptr()
        assert _guards_intact(obuf, out_bytes), "output guard overwritten"
        assert _guards_intact(wbuf, need), "workspace guard overwritten"
        assert torch.equal(got, ref)
