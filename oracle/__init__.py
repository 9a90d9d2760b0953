"""CPU oracle for paged single-token decode attention -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, fp64 restatement of what the paged-KV decode path
computes. It exists so that the CUDA library can be checked against something
obviously correct. Only the test-suite, the smoke check in ``__graft_entry__`` and
the CPU-baseline leg of ``bench.py`` may import it; the product path (the C-ABI
library and its Python binding) never does, and it shares no code with it.

Sources (the pages the method is taken from):

* "大模型工程（五）：推理优化核心技法" (chenk.top, LLM engineering part 5), sections
  "两个特性截然不同的阶段" (decode reads the whole KV cache every step),
  "分页注意力" (fixed 16-token blocks, per-request block table, the 47/200-token
  worked example, at most 15 tokens wasted, prefix sharing), "块管理器：分页如何运作"
  (free list, refcounted copy-on-write blocks, eviction of a request's blocks to
  pinned host memory and back), "INT8 仅权重量化" (``w_q = round(w/s)``), "FP8（及
  H100/H200 硬件路径）" (E4M3 and E5M2, E5M2 for KV caches), "KV 缓存量化"
  (per-token-per-head scales) and "推测解码" (the target model scores k drafted
  tokens plus one in a single pass: multi-query decode).
* The gsyq.cn inference-optimisation page, section 2.1 (the KV-cache size formula and
  its 7B example), 2.2 (block sizes 16 or 32, shared blocks) and 2.3 (per-token or
  per-channel KV scales, softmax stability after quantisation).

Every function here is pinned against the pages' worked examples, closed forms,
invariants, independent implementations and brute force -- ``tests/test_oracle_pins.py``
(paging, decode, INT8), ``tests/test_oracle_fp8_pins.py``, ``tests/test_oracle_multi_pins.py``
and ``tests/test_oracle_block_pins.py`` (copy-on-write and swap); none is marked
"parity unpinned".
"""

from .paged_attention import (  # noqa: F401
    num_blocks_for,
    kv_cache_bytes,
    append_scatter,
    quantize_rows_int8,
    dequantize_rows_int8,
    append_scatter_int8,
    gather_sequence,
    gather_sequence_int8,
    attend_one_head,
    decode_attention,
    decode_attention_int8,
    decode_attention_multi,
    decode_attention_multi_quantized,
    FP8_MAX,
    fp8_decode,
    fp8_round,
    quantize_rows_fp8,
    dequantize_rows_fp8,
    append_scatter_fp8,
    gather_sequence_fp8,
    decode_attention_fp8,
    copy_blocks,
    swap_out_blocks,
    swap_in_blocks,
)
