"""The C-ABI library builds, loads, and exports every entry point the public header
declares; host-side argument checks answer without touching a GPU."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib_path():
    from paged_kv_decode_02_gb300 import build_lib
    try:
        build_lib._nvcc()
    except RuntimeError as e:  # no CUDA toolkit on this machine
        pytest.skip(str(e))
    return build_lib.build()   # a compile error fails the test


def test_header_declares_the_api():
    names = _declared_functions()
    for must in ("pkv_append_bf16", "pkv_append_int8", "pkv_decode_bf16", "pkv_decode_int8",
                 "pkv_decode_workspace_bytes", "pkv_status_string", "pkv_version"):
        assert must in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(re.findall(r"\bT (pkv_\w+)", out.stdout))
        assert set(_declared_functions()) <= exported


def test_binding_signatures_cover_the_header(lib_path):
    from paged_kv_decode_02_gb300 import pagedkv
    assert set(pagedkv.EXPORTS) == set(_declared_functions())
    lib = pagedkv.load_library(lib_path)
    assert lib.pkv_version() == 100
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert b"NULL" in lib.pkv_status_string(-1)
    assert lib.pkv_status_string(12345) == b"unknown pkv_status"
    assert b"pinned" in lib.pkv_status_string(-8)


def test_host_validation_without_gpu(lib_path):
    """Each failing check returns before any CUDA call, so these run on a CPU machine."""
    from paged_kv_decode_02_gb300 import pagedkv
    lib = pagedkv.load_library(lib_path)
    launches_before = lib.pkv_kernel_launch_count()
    good = pagedkv.Dims(4, 8, 8, 64, 16, 64, 4)
    p = ctypes.c_void_p(0x1000)
    st = lib.pkv_decode_bf16(None, p, p, p, p, p, 0.1, ctypes.byref(good), p, 1 << 20, None, None)
    assert st == pagedkv.Status.ERR_NULL
    bad_bs = pagedkv.Dims(4, 8, 8, 64, 24, 64, 4)
    st = lib.pkv_decode_bf16(p, p, p, p, p, p, 0.1, ctypes.byref(bad_bs), p, 1 << 20, None, None)
    assert st == pagedkv.Status.ERR_UNSUPPORTED
    bad_d = pagedkv.Dims(4, 8, 8, 96, 16, 64, 4)
    st = lib.pkv_decode_bf16(p, p, p, p, p, p, 0.1, ctypes.byref(bad_d), p, 1 << 20, None, None)
    assert st == pagedkv.Status.ERR_UNSUPPORTED
    bad_group = pagedkv.Dims(4, 6, 4, 64, 16, 64, 4)
    st = lib.pkv_decode_bf16(p, p, p, p, p, p, 0.1, ctypes.byref(bad_group), p, 1 << 20, None,
                             None)
    assert st == pagedkv.Status.ERR_SHAPE
    st = lib.pkv_decode_bf16(p, p, p, p, p, p, 0.1, None, p, 1 << 20, None, None)
    assert st == pagedkv.Status.ERR_NULL
    mis = ctypes.c_void_p(0x1008)
    st = lib.pkv_decode_bf16(mis, p, p, p, p, p, 0.1, ctypes.byref(good), p, 1 << 20, None, None)
    assert st == pagedkv.Status.ERR_ALIGNMENT
    st = lib.pkv_decode_int8(p, p, p, p, None, p, p, p, 0.1, ctypes.byref(good), p, 1 << 20, None,
                             None)
    assert st == pagedkv.Status.ERR_NULL
    st = lib.pkv_append_bf16(p, None, p, p, p, 3, ctypes.byref(good), None)
    assert st == pagedkv.Status.ERR_NULL
    st = lib.pkv_append_bf16(p, p, p, p, p, -1, ctypes.byref(good), None)
    assert st == pagedkv.Status.ERR_SHAPE
    st = lib.pkv_append_bf16(None, None, None, None, None, 0, ctypes.byref(good), None)
    assert st == pagedkv.Status.OK          # zero tokens: no-op
    st = lib.pkv_append_int8(p, p, p, p, None, p, p, 3, ctypes.byref(good), None)
    assert st == pagedkv.Status.ERR_NULL
    # FP8 entry points take only the two FP8 format codes
    st = lib.pkv_decode_fp8(p, p, p, p, p, p, p, p, 0.1, pagedkv.KV_INT8, ctypes.byref(good), p,
                            1 << 20, None, None)
    assert st == pagedkv.Status.ERR_DTYPE
    st = lib.pkv_decode_fp8(p, p, p, p, None, p, p, p, 0.1, pagedkv.KV_FP8_E5M2,
                            ctypes.byref(good), p, 1 << 20, None, None)
    assert st == pagedkv.Status.ERR_NULL
    st = lib.pkv_append_fp8(p, p, p, p, p, p, p, 3, pagedkv.KV_BF16, ctypes.byref(good), None)
    assert st == pagedkv.Status.ERR_DTYPE
    st = lib.pkv_append_fp8(p, p, p, p, None, p, p, 3, pagedkv.KV_FP8_E4M3, ctypes.byref(good),
                            None)
    assert st == pagedkv.Status.ERR_NULL
    # block moves: argument checks before any CUDA call
    st = lib.pkv_copy_blocks(p, p, None, None, None, p, 4, pagedkv.KV_BF16, ctypes.byref(good),
                             None, None)
    assert st == pagedkv.Status.ERR_NULL
    st = lib.pkv_copy_blocks(p, p, None, None, p, p, 4, 9, ctypes.byref(good), None, None)
    assert st == pagedkv.Status.ERR_DTYPE
    st = lib.pkv_copy_blocks(p, p, None, None, p, p, 0, pagedkv.KV_BF16, ctypes.byref(good),
                             None, None)
    assert st == pagedkv.Status.OK
    st = lib.pkv_copy_blocks(p, p, None, None, p, p, 4, pagedkv.KV_INT8, ctypes.byref(good),
                             None, None)
    assert st == pagedkv.Status.ERR_NULL                  # one-byte caches need scales
    st = lib.pkv_swap_out(None, p, p, p, p, p, p, p, p, 4, pagedkv.KV_INT8, ctypes.byref(good),
                          None, None)
    assert st == pagedkv.Status.ERR_NULL
    st = lib.pkv_swap_in(p, mis, None, None, p, p, None, None, p, 4, pagedkv.KV_BF16,
                         ctypes.byref(good), None, None)
    assert st == pagedkv.Status.ERR_ALIGNMENT
    n = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(good), 4, ctypes.byref(n)) == \
        pagedkv.Status.ERR_DTYPE
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(good), 7, ctypes.byref(n)) == \
        pagedkv.Status.ERR_DTYPE
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(good), 0, None) == pagedkv.Status.ERR_NULL
    # multi-query decode: 1 <= q_len <= PKV_MAX_QUERY_LEN (256)
    for q_len in (0, 257):
        assert lib.pkv_decode_multi_workspace_bytes(ctypes.byref(good), q_len,
                                                    ctypes.byref(n)) == pagedkv.Status.ERR_SHAPE
        st = lib.pkv_decode_multi_bf16(p, p, p, p, p, p, q_len, 0.1, ctypes.byref(good), p,
                                       1 << 20, None, None)
        assert st == pagedkv.Status.ERR_SHAPE
    assert lib.pkv_decode_multi_workspace_bytes(ctypes.byref(good), 2, None) == \
        pagedkv.Status.ERR_NULL
    st = lib.pkv_decode_multi_bf16(p, p, p, None, p, p, 2, 0.1, ctypes.byref(good), p, 1 << 20,
                                   None, None)
    assert st == pagedkv.Status.ERR_NULL
    # cascade: the shared prefix is 1 .. max_blocks_per_seq blocks
    for blocks in (0, 5):
        assert lib.pkv_decode_cascade_workspace_bytes(ctypes.byref(good), blocks,
                                                      ctypes.byref(n)) == pagedkv.Status.ERR_SHAPE
    st = lib.pkv_decode_cascade_bf16(p, mis, p, p, p, p, 2, 0.1, ctypes.byref(good), p, 1 << 20,
                                     None, None)
    assert st == pagedkv.Status.ERR_ALIGNMENT
    st = lib.pkv_decode_cascade_bf16(p, p, p, p, p, p, 2, 0.1, ctypes.byref(bad_bs), p, 1 << 20,
                                     None, None)
    assert st == pagedkv.Status.ERR_UNSUPPORTED
    # nothing above reached a launch
    assert lib.pkv_kernel_launch_count() == launches_before


def test_binding_host_checks_without_gpu():
    """The binding's own checks (the C ABI cannot see buffer sizes) refuse
    disagreeing shapes, unusable workspaces and status words, and host buffers too
    short for a swap, before any library call."""
    import torch
    from paged_kv_decode_02_gb300 import pagedkv as P
    kc = torch.zeros(6, 2, 16, 64, dtype=torch.bfloat16)
    row = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    slots = torch.zeros(3, dtype=torch.int64)
    P._append_shapes(row, row, kc, kc.clone(), slots)                   # consistent: passes
    for args in ((row[:2], row, kc, kc, slots),                          # k rows vs slots
                 (row, row, kc, kc, slots[:2]),                          # short slot_mapping
                 (row[..., :32], row[..., :32], kc, kc, slots),          # head_dim
                 (row, row, kc, kc[:5], slots)):                         # v_cache pool
        with pytest.raises(ValueError):
            P._append_shapes(*args)
    sc = torch.zeros(6, 2, 16)
    P._cache_shapes(kc, kc, sc, sc)
    with pytest.raises(ValueError):
        P._cache_shapes(kc, kc, sc, sc[:, :, :8])                       # scales per block
    dev = torch.device("cuda", 0)
    with pytest.raises(ValueError):
        P._workspace(torch.zeros(1 << 10, dtype=torch.uint8), 256, dev)   # host memory
    with pytest.raises(ValueError):
        P._status_word(torch.zeros(1, dtype=torch.int32), dev)          # host memory
    assert P._status_word(None, dev) is None
    with pytest.raises(ValueError):                                       # not pinned
        P._host_buffers(P.KV_BF16, 3, 4096, 0, torch.zeros(3, 4096, dtype=torch.uint8),
                        torch.zeros(3, 4096, dtype=torch.uint8), None, None)
